// Flash decoding: a few query rows per (batch, head) against a long KV cache.
//
// Follows "Flash decoding" (linear algebra for programmers, part 4),
// "Overview of the algorithm": the keys are split into n_splits chunks; the
// split kernel runs the online softmax over one chunk and writes the
// unnormalised partial (O_s, m_s, l_s); the combine kernel rescales every
// partial by e^{m_s - m_g} and divides once by l_g.
//
// GB300 design (not the page's): the split kernel is HBM-bound (one FMA per
// byte), so each CTA streams its chunk of K and V through a 3-stage ring of
// shared-memory buffers filled by bulk TMA copies (cp.async.bulk, one producer
// warp, L2 evict-first), and 4 compute warps read 16-byte vectors from it.
// A "row unit" of D*size/16 lanes owns one key at a time; each unit carries
// its own (m, l, acc) online-softmax state in registers, and the units of the
// CTA are merged with the (m, l) monoid at the end ("Flash Attention" notes,
// "Deriving the online softmax").
//
// Several query rows (R <= 4) of one (batch, head) share the cache: each K and V
// vector a lane unpacks serves all of them, so the HBM traffic stays that of
// one row. Row r of head bh is partial row bh*R + r, so the combine runs over
// B*H*R rows unchanged; it also writes LSE = m_g + ln l_g when asked.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecWarps = 4;                      // compute warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecStages = 3;
constexpr int kDecStageBytes = 16384;              // K + V bytes per stage
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int DT>
struct Elem;
template <>
struct Elem<kF32> {
  using T = float;
  static constexpr int kSize = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static T from_f32(float x) { return x; }
};
template <>
struct Elem<kF16> {
  using T = __half;
  static constexpr int kSize = 2;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static T from_f32(float x) { return __float2half_rn(x); }
};
template <>
struct Elem<kBF16> {
  using T = __nv_bfloat16;
  static constexpr int kSize = 2;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static T from_f32(float x) { return __float2bfloat16_rn(x); }
};

template <int D, int DT>
struct DecCfg {
  static constexpr int kES = Elem<DT>::kSize;
  static constexpr int kRow = D * kES;             // bytes per key row
  static constexpr int kLPK = kRow / 16;           // lanes per key (one 16-byte vector each)
  static constexpr int kKPW = 32 / kLPK;           // keys per warp in parallel
  static constexpr int kEPL = 16 / kES;            // elements per lane
  static constexpr int kNU = kDecWarps * kKPW;     // row units per CTA
  static constexpr int kTK = kDecStageBytes / (2 * kRow);  // keys per stage
  static constexpr int kG = kTK / kNU;             // keys per row unit per stage
  static_assert(kLPK >= 1 && kLPK <= 32 && kG >= 1, "decode tiling");
};

struct DecSmemHdr {
  unsigned long long full[kDecStages];
  unsigned long long empty[kDecStages];
  int abort_flag;
};

// R: query rows held per thread (template); rows <= R of them are real (q, ws hold `rows`).
template <int D, int DT, int R>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const typename Elem<DT>::T* __restrict__ q,
                                                                   const typename Elem<DT>::T* __restrict__ K,
                                                                   const typename Elem<DT>::T* __restrict__ V,
                                                                   float* __restrict__ ws, int BH, int rows, int N,
                                                                   int n_splits, float scale_log2,
                                                                   DevStatus* status,
                                                                   unsigned long long budget_ns, int inject) {
  using C = DecCfg<D, DT>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecSmemHdr* hdr = reinterpret_cast<DecSmemHdr*>(smem_raw);
  uint8_t* ring = smem_raw + 128;  // stage st: K at ring + st*kDecStageBytes, V right after K
  // merge scratch: the ring itself, once every compute warp has read its last stage (saves the
  // shared memory that would cost a resident CTA per SM with several rows)
  float* red = reinterpret_cast<float*>(ring);

  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int chunk = (N + n_splits - 1) / n_splits;
  const int n_start = min(split * chunk, N);
  const int n_end = min(n_start + chunk, N);
  const int nkeys = n_end - n_start;
  const int nstage = (nkeys + C::kTK - 1) / C::kTK;

  // partial of query row r of this head (row bh*rows + r of the combine)
  const size_t nrow = static_cast<size_t>(BH) * rows;
  auto ws_O = [&](int r) { return ws + ((static_cast<size_t>(bh) * rows + r) * n_splits + split) * D; };
  auto ws_m = [&](int r) { return ws + nrow * n_splits * D + (static_cast<size_t>(bh) * rows + r) * n_splits + split; };
  auto ws_l = [&](int r) { return ws_m(r) + nrow * n_splits; };

  if (nkeys <= 0) {  // empty split: the identity of the merge
    for (int i = threadIdx.x; i < rows * D; i += blockDim.x) ws_O(i / D)[i % D] = 0.f;
    if (threadIdx.x < rows) {
      *ws_m(threadIdx.x) = -INFINITY;
      *ws_l(threadIdx.x) = 0.f;
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&hdr->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->empty[s]), kDecWarps);
    }
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernDecodeSplit};

  const size_t head_off = static_cast<size_t>(bh) * N * D;

  if (warp == kDecWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      const char* kb = reinterpret_cast<const char*>(K + head_off);
      const char* vb = reinterpret_cast<const char*>(V + head_off);
      int issued = 0;
      // test-only fault injection: the first CTA never fills its first stage, so its consumers'
      // bounded wait runs out and the launch reports a timeout (no fault, no trap)
      const bool skip_first = inject == kInjectDecodeStage && blockIdx.x == 0 && blockIdx.y == 0;
      for (int it = 0; it < nstage; ++it) {
        const int st = it % kDecStages;
        const uint32_t ph = static_cast<uint32_t>(it / kDecStages) & 1u;
        if (it == 0 && skip_first) {
          issued = 1;
          continue;
        }
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ph ^ 1u, wc, 1)) break;
        const int k0 = n_start + it * C::kTK;
        const int nk = min(C::kTK, n_end - k0);
        const uint32_t bytes = static_cast<uint32_t>(nk) * C::kRow;
        const uint32_t full = ptx::smem_u32(&hdr->full[st]);
        ptx::mbar_arrive_expect_tx(full, 2u * bytes);
        uint8_t* sk = ring + st * kDecStageBytes;
        ptx::bulk_load(ptx::smem_u32(sk), kb + static_cast<size_t>(k0) * C::kRow, bytes, full, pol);
        ptx::bulk_load(ptx::smem_u32(sk + kDecStageBytes / 2), vb + static_cast<size_t>(k0) * C::kRow, bytes, full,
                       pol);
        issued = it + 1;
      }
      if (hdr->abort_flag) {  // let copies already in flight land before the CTA exits
        for (int it = max(0, issued - kDecStages); it < issued; ++it)
          if (!(it == 0 && skip_first))
            ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[it % kDecStages]),
                                 static_cast<uint32_t>(it / kDecStages) & 1u, 100000000ull);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int ru = warp * C::kKPW + lane / C::kLPK;  // row unit
  const int sl = lane % C::kLPK;                   // 16-byte slot within the key row
  float qv[R][C::kEPL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < rows) {
      const uint4 u = *reinterpret_cast<const uint4*>(
          reinterpret_cast<const char*>(q + (static_cast<size_t>(bh) * rows + r) * D) + sl * 16);
      Elem<DT>::unpack(u, qv[r]);
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) qv[r][e] *= scale_log2;  // scores come out in log2 units
    } else {
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) qv[r][e] = 0.f;  // a padding row: computed, never written
    }
  }
  // several rows: lane offsets of the butterfly and the lane (within the key's group) that ends
  // up holding row r; with R > 1, m[0] and l[0] are the state of this lane's row my_row
  constexpr int kO1 = C::kLPK / 2, kO2 = C::kLPK / 4;
  static_assert(R == 1 || R == 2 || (R == 4 && kO2 >= 1), "decode rows");
  auto row_lane = [](int r) { return R == 4 ? (r >> 1) * kO1 + (r & 1) * kO2 : r * kO1; };
  const int group0 = lane - sl;  // first lane of this key's group
  const int my_row = R == 1 ? 0 : (R == 2 ? ((sl & kO1) ? 1 : 0) : ((sl & kO1) ? 2 : 0) + ((sl & kO2) ? 1 : 0));
  float m[R], l[R];
  float acc[R][C::kEPL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < C::kEPL; ++e) acc[r][e] = 0.f;
  }

  for (int it = 0; it < nstage; ++it) {
    const int st = it % kDecStages;
    const uint32_t ph = static_cast<uint32_t>(it / kDecStages) & 1u;
    if (!ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), ph, wc, 2)) break;
    const int nk = min(C::kTK, n_end - (n_start + it * C::kTK));
    const uint8_t* sk = ring + st * kDecStageBytes;
    const uint8_t* sv = sk + kDecStageBytes / 2;

    if constexpr (R == 1) {
      float s[C::kG][R];
  #pragma unroll
      for (int g = 0; g < C::kG; ++g) {
        const int kk = ru + g * C::kNU;
        float part[R];
  #pragma unroll
        for (int r = 0; r < R; ++r) part[r] = 0.f;
        if (kk < nk) {
          float kf[C::kEPL];
          Elem<DT>::unpack(*reinterpret_cast<const uint4*>(sk + kk * C::kRow + sl * 16), kf);
  #pragma unroll
          for (int r = 0; r < R; ++r)
  #pragma unroll
            for (int e = 0; e < C::kEPL; ++e) part[r] = fmaf(qv[r][e], kf[e], part[r]);
        }
  #pragma unroll
        for (int r = 0; r < R; ++r) {
  #pragma unroll
          for (int o = C::kLPK / 2; o >= 1; o >>= 1) part[r] += __shfl_xor_sync(0xFFFFFFFFu, part[r], o);
          s[g][r] = kk < nk ? part[r] : -INFINITY;
        }
      }
      float p[C::kG][R];
  #pragma unroll
      for (int r = 0; r < R; ++r) {
        float mb = s[0][r];
  #pragma unroll
        for (int g = 1; g < C::kG; ++g) mb = fmaxf(mb, s[g][r]);
        const float m_new = fmaxf(m[r], mb);
        const float m_safe = m_new == -INFINITY ? 0.f : m_new;
        const float corr = ptx::ex2(m[r] - m_safe);
        float ps = 0.f;
  #pragma unroll
        for (int g = 0; g < C::kG; ++g) {
          p[g][r] = ptx::ex2(s[g][r] - m_safe);
          ps += p[g][r];
        }
        l[r] = fmaf(l[r], corr, ps);
        m[r] = m_new;
  #pragma unroll
        for (int e = 0; e < C::kEPL; ++e) acc[r][e] *= corr;
      }
  #pragma unroll
      for (int g = 0; g < C::kG; ++g) {
        const int kk = ru + g * C::kNU;
        if (kk < nk) {
          float vf[C::kEPL];
          Elem<DT>::unpack(*reinterpret_cast<const uint4*>(sv + kk * C::kRow + sl * 16), vf);
  #pragma unroll
          for (int r = 0; r < R; ++r)
  #pragma unroll
            for (int e = 0; e < C::kEPL; ++e) acc[r][e] = fmaf(p[g][r], vf[e], acc[r][e]);
        }
      }
    } else {
      // Several rows: a reduce-scatter butterfly over the key's lanes leaves each lane the full
      // score of one row (my_row), so the online softmax runs once per lane; the weights are then
      // broadcast from the lanes holding each row for the accumulator update. Every shuffle runs
      // on all 32 lanes (kk differs between the key groups of a warp).
      float sc[C::kG];
#pragma unroll
      for (int g = 0; g < C::kG; ++g) {
        const int kk = ru + g * C::kNU;
        float part[R];
#pragma unroll
        for (int r = 0; r < R; ++r) part[r] = 0.f;
        if (kk < nk) {
          float kf[C::kEPL];
          Elem<DT>::unpack(*reinterpret_cast<const uint4*>(sk + kk * C::kRow + sl * 16), kf);
          // pairs of elements on the f32x2 FMA (half the instructions: this path is issue-bound)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < C::kEPL; e += 2)
              p2 = ptx::ffma2(make_float2(qv[r][e], qv[r][e + 1]), make_float2(kf[e], kf[e + 1]), p2);
            part[r] = p2.x + p2.y;
          }
        }
        float c;
        if constexpr (R == 2) {
          const bool hi = (sl & kO1) != 0;
          c = (hi ? part[1] : part[0]) + __shfl_xor_sync(0xFFFFFFFFu, hi ? part[0] : part[1], kO1);
#pragma unroll
          for (int o = kO1 / 2; o >= 1; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
        } else {
          const bool hi = (sl & kO1) != 0, lo = (sl & kO2) != 0;
          const float a0 = (hi ? part[2] : part[0]) + __shfl_xor_sync(0xFFFFFFFFu, hi ? part[0] : part[2], kO1);
          const float a1 = (hi ? part[3] : part[1]) + __shfl_xor_sync(0xFFFFFFFFu, hi ? part[1] : part[3], kO1);
          c = (lo ? a1 : a0) + __shfl_xor_sync(0xFFFFFFFFu, lo ? a0 : a1, kO2);
#pragma unroll
          for (int o = kO2 / 2; o >= 1; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
        }
        sc[g] = kk < nk ? c : -INFINITY;
      }
      float mb = sc[0];
#pragma unroll
      for (int g = 1; g < C::kG; ++g) mb = fmaxf(mb, sc[g]);
      const float m_new = fmaxf(m[0], mb);
      const float m_safe = m_new == -INFINITY ? 0.f : m_new;
      const float corr = ptx::ex2(m[0] - m_safe);
      float pw[C::kG];
      float ps = 0.f;
#pragma unroll
      for (int g = 0; g < C::kG; ++g) {
        pw[g] = ptx::ex2(sc[g] - m_safe);
        ps += pw[g];
      }
      l[0] = fmaf(l[0], corr, ps);  // this lane's row
      m[0] = m_new;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float cr = __shfl_sync(0xFFFFFFFFu, corr, group0 + row_lane(r));
#pragma unroll
        for (int e = 0; e < C::kEPL; e += 2) {
          const float2 a = ptx::fmul2(make_float2(acc[r][e], acc[r][e + 1]), make_float2(cr, cr));
          acc[r][e] = a.x;
          acc[r][e + 1] = a.y;
        }
      }
#pragma unroll
      for (int g = 0; g < C::kG; ++g) {
        const int kk = ru + g * C::kNU;
        float pr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) pr[r] = __shfl_sync(0xFFFFFFFFu, pw[g], group0 + row_lane(r));
        if (kk < nk) {
          float vf[C::kEPL];
          Elem<DT>::unpack(*reinterpret_cast<const uint4*>(sv + kk * C::kRow + sl * 16), vf);
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < C::kEPL; e += 2) {
              const float2 a = ptx::ffma2(make_float2(pr[r], pr[r]), make_float2(vf[e], vf[e + 1]),
                                          make_float2(acc[r][e], acc[r][e + 1]));
              acc[r][e] = a.x;
              acc[r][e + 1] = a.y;
            }
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->empty[st]));
  }

  // Merge the row units of this CTA: (m, l) monoid per query row, then write the partials.
  float* red_m = red;                     // [kNU][R]
  float* red_l = red + C::kNU * R;        // [kNU][R]
  float* red_acc = red + 2 * C::kNU * R;  // [kNU][R][D]
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");  // the ring is no longer read
  if (R == 1) {
    if (sl == 0) {
      red_m[ru] = m[0];
      red_l[ru] = l[0];
    }
  } else if (sl == row_lane(my_row)) {  // one lane per row holds its (m, l)
    red_m[ru * R + my_row] = m[0];
    red_l[ru * R + my_row] = l[0];
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int e = 0; e < C::kEPL; ++e) red_acc[(ru * R + r) * D + sl * C::kEPL + e] = acc[r][e];
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
  if (hdr->abort_flag) return;

  for (int i = threadIdx.x; i < rows * D; i += kDecWarps * 32) {
    const int r = i / D, d = i - r * D;
    float mg = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::kNU; ++u) mg = fmaxf(mg, red_m[u * R + r]);
    const float mg_safe = mg == -INFINITY ? 0.f : mg;
    float o = 0.f;
#pragma unroll
    for (int u = 0; u < C::kNU; ++u) o = fmaf(ptx::ex2(red_m[u * R + r] - mg_safe), red_acc[(u * R + r) * D + d], o);
    ws_O(r)[d] = o;
  }
  if (threadIdx.x < rows) {
    const int r = threadIdx.x;
    float mg = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::kNU; ++u) mg = fmaxf(mg, red_m[u * R + r]);
    const float mg_safe = mg == -INFINITY ? 0.f : mg;
    float lg = 0.f;
#pragma unroll
    for (int u = 0; u < C::kNU; ++u) lg = fmaf(ptx::ex2(red_m[u * R + r] - mg_safe), red_l[u * R + r], lg);
    *ws_m(r) = mg * kLn2;  // natural-log units, as in the page's equations (-inf stays -inf)
    *ws_l(r) = lg;
  }
}

constexpr int kCombThreads = 128;
constexpr int kCombChunk = 1024;

template <int D, int DT>
// One CTA per query row (B*H*R of them, row-major like O); LSE may be null.
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const float* __restrict__ ws,
                                                                      typename Elem<DT>::T* __restrict__ O,
                                                                      float* __restrict__ LSE, int BH,
                                                                      int n_splits) {
  __shared__ float w[kCombChunk];
  __shared__ float red[kCombThreads / 32];
  __shared__ float s_mg, s_lg;
  const int bh = blockIdx.x;
  const float* Os = ws + static_cast<size_t>(bh) * n_splits * D;
  const float* ms = ws + static_cast<size_t>(BH) * n_splits * D + static_cast<size_t>(bh) * n_splits;
  const float* ls = ms + static_cast<size_t>(BH) * n_splits;
  const int tid = threadIdx.x;

  // PDL: wait until the split kernel's partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float mx = -INFINITY;
  for (int s = tid; s < n_splits; s += kCombThreads) mx = fmaxf(mx, ms[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    float v = red[0];
    for (int i = 1; i < kCombThreads / 32; ++i) v = fmaxf(v, red[i]);
    s_mg = v;
  }
  __syncthreads();
  const float mg = s_mg;

  float lsum = 0.f, o = 0.f;
  for (int c0 = 0; c0 < n_splits; c0 += kCombChunk) {
    const int cn = min(kCombChunk, n_splits - c0);
    for (int s = tid; s < cn; s += kCombThreads) {
      const float ww = ptx::ex2((ms[c0 + s] - mg) * kLog2e);  // e^{m_s - m_g}; empty split -> 0
      w[s] = ww;
      lsum = fmaf(ww, ls[c0 + s], lsum);
    }
    __syncthreads();
    if (tid < D)
      for (int s = 0; s < cn; ++s) o = fmaf(w[s], Os[static_cast<size_t>(c0 + s) * D + tid], o);
    __syncthreads();
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, off);
  if ((tid & 31) == 0) red[tid >> 5] = lsum;
  __syncthreads();
  if (tid == 0) {
    float v = 0.f;
    for (int i = 0; i < kCombThreads / 32; ++i) v += red[i];
    s_lg = v;
  }
  __syncthreads();
  if (tid < D) O[static_cast<size_t>(bh) * D + tid] = Elem<DT>::from_f32(o / s_lg);
  if (LSE != nullptr && tid == 0) LSE[bh] = mg + logf(s_lg);  // natural log, like the forward's LSE
}

template <int D, int DT, int R>
cudaError_t launch_decode_t(const void* q, const void* K, const void* V, void* O, float* LSE, float* ws, int BH,
                            int rows, int N, float scale, int n_splits, const LaunchCtx& ctx) {
  using C = DecCfg<D, DT>;
  using T = typename Elem<DT>::T;
  constexpr size_t kRed = (2 * C::kNU * R + C::kNU * R * D) * sizeof(float);  // merge scratch, over the ring
  static_assert(kRed <= static_cast<size_t>(kDecStages) * kDecStageBytes, "decode merge scratch");
  const size_t smem = 128 + static_cast<size_t>(kDecStages) * kDecStageBytes;
  auto kern = decode_split_kernel<D, DT, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(n_splits, BH);
  kern<<<grid, kDecThreads, smem, ctx.stream>>>(static_cast<const T*>(q), static_cast<const T*>(K),
                                                static_cast<const T*>(V), ws, BH, rows, N, n_splits, scale * kLog2e,
                                                ctx.status, ctx.wait_budget_ns, ctx.inject);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(BH * rows);
  cfg.blockDim = dim3(kCombThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, DT>, static_cast<const float*>(ws), static_cast<T*>(O),
                            LSE, BH * rows, n_splits);
}

}  // namespace

cudaError_t launch_decode(const void* q, const void* K, const void* V, void* O, float* LSE, float* ws, int BH,
                          int rows, int N, int D, float scale, int n_splits, int dtype, const LaunchCtx& ctx) {
  if (BH > 65535) return cudaErrorNotSupported;  // grid.y limit of the split kernel
  if (rows < 1 || rows > kDecMaxRows) return cudaErrorNotSupported;
  // query rows held per thread: 1, 2 or 4 (three rows run the four-row kernel with one padding row)
#define FA_DEC(DD, TT)                                                                                   \
  if (D == DD && dtype == TT) {                                                                          \
    if (rows == 1) return launch_decode_t<DD, TT, 1>(q, K, V, O, LSE, ws, BH, rows, N, scale, n_splits, ctx); \
    if (rows == 2) return launch_decode_t<DD, TT, 2>(q, K, V, O, LSE, ws, BH, rows, N, scale, n_splits, ctx); \
    return launch_decode_t<DD, TT, 4>(q, K, V, O, LSE, ws, BH, rows, N, scale, n_splits, ctx);             \
  }
  FA_DEC(64, kF32)
  FA_DEC(64, kF16)
  FA_DEC(64, kBF16)
  FA_DEC(128, kF32)
  FA_DEC(128, kF16)
  FA_DEC(128, kBF16)
#undef FA_DEC
  return cudaErrorNotSupported;
}

}  // namespace fa
