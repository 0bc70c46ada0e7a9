// Forward prefill for f32 inputs and outputs (D = 64), 3xTF32 on tcgen05.
//
// Same method as the half-precision forward ("Flash attention, f32", Phobos
// examples): one block of 128 query rows per CTA, keys walked in blocks with a
// running max, denominator and unnormalised accumulator, one division at the
// end; LSE = m + log l ("06: Fused attention"). The page's kernel rounds its f32
// operands to f16 for the tensor cores; that misses an f32 tolerance, so here
// every product is split: x = hi + lo with hi = x rounded to tf32 (cvt.rna) and
// lo = x - hi, and A B ~= Ah Bh + Al Bh + Ah Bl with f32 accumulation
// (kind::tf32, 8-element k-steps). hi has zero low mantissa bits, so the result
// does not depend on how the tensor core reduces f32 to tf32.
//
// GB300 layout: one CTA per 128-row tile of one (batch, head); a producer warp
// streams 64-key blocks of K and V (f32, 128-byte swizzle) through a two-stage
// ring; four split warps rewrite each landed K block in place as its hi part
// and write its lo part next to it (and Q's, once per tile), and write V
// transposed, as hi and lo, because the tf32 MMA reads its B operand K-major
// only (an MN-major tf32 operand was measured to read as zeros); one MMA thread
// issues S = Q K^T (3 groups) and O += P V (3 groups); four softmax warps (one
// row per thread) write P's hi part over S and its lo part beside it in
// tensor memory.
// The tensor core's f32 accumulation was measured to lose about one unit in the
// last place per add, always towards zero: a chain of ~1500 adds (64 key blocks x
// 24 MMAs) into one accumulator biased O by ~3e-5. So each key block's P V starts
// from zero in tensor memory (24 adds) and the softmax threads sum the block
// partials in registers with round-to-nearest adds; the rescale of O happens
// there too.
// Tensor memory: S / P_hi [0,64), P_lo [64,128), block partial of O [128,192).
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM32 = 128;          // query rows per CTA
constexpr int kBN32 = 64;           // keys per block
constexpr int kD32 = 64;
constexpr int kRowB = 128;          // bytes per swizzled row (32 f32)
constexpr int kQChunk = kBM32 * kRowB;    // 16 KB: 128 rows x 32 columns
constexpr int kKChunk = kBN32 * kRowB;    // 8 KB: 64 rows x 32 columns
constexpr int kQBytes = 2 * kQChunk;      // 64 columns
constexpr int kKBytes = 2 * kKChunk;
constexpr int kStages32 = 2;
constexpr int kThreads32 = 320;     // softmax 0-3, split 4-7, producer 8, MMA 9
constexpr int kWarpProd32 = 8, kWarpMma32 = 9;
constexpr float kLog2e32 = 1.4426950408889634f;
constexpr float kLn2_32 = 0.6931471805599453f;
constexpr int kF32Slot = kF32SlotFloats;

struct F32Hdr {
  unsigned long long q_full, q_split, q_empty;
  unsigned long long kv_full[kStages32], kv_split[kStages32], kv_empty[kStages32];
  unsigned long long s_full, p_full, o_full, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// smem layout (1024-aligned): Qhi, Qlo, then per stage: Khi, Klo, V (as loaded), V^T hi, V^T lo
constexpr int kSmem32 = 1024 + 1024 + 2 * kQBytes + kStages32 * 5 * kKBytes;
static_assert(kSmem32 <= 232448, "shared memory budget");

__device__ __forceinline__ float tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Rewrites `n16` 16-byte vectors at generic address `hi` in place as their tf32
// hi parts and writes the lo parts at `lo`; threads [tid0, tid0 + nthreads).
__device__ __forceinline__ void split_block(float4* hi, float4* lo, int n16, int tid, int nthreads) {
  for (int i = tid; i < n16; i += nthreads) {
    const float4 x = hi[i];
    const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
    hi[i] = h;
    lo[i] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  }
}

// Byte offset of element (row, col) in a tile of 128-byte-swizzled rows split
// into 32-column chunks of `chunk` bytes (the TMA SWIZZLE_128B layout): the
// 16-byte unit index within a row is XORed with row % 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, uint32_t chunk) {
  const int c = col & 31;
  return (col >> 5) * chunk + row * kRowB + ((((c >> 2) ^ (row & 7)) << 4) | ((c & 3) << 2));
}

// V block [64 keys x 64 d] as loaded -> V^T [64 d x 64 keys], split into tf32
// hi and lo, in the K-major swizzled layout the PV MMA reads.
__device__ __forceinline__ void split_transpose_v(const float* v, float* vth, float* vtl, int tid, int nthreads) {
  const uint8_t* src = reinterpret_cast<const uint8_t*>(v);
  uint8_t* dh = reinterpret_cast<uint8_t*>(vth);
  uint8_t* dl = reinterpret_cast<uint8_t*>(vtl);
  for (int e = tid; e < kBN32 * kD32; e += nthreads) {
    const int key = e / kD32, d = e % kD32;
    const float x = *reinterpret_cast<const float*>(src + sw128_offset(key, d, kKChunk));
    const float h = tf32_hi(x);
    const uint32_t o = sw128_offset(d, key, kKChunk);
    *reinterpret_cast<float*>(dh + o) = h;
    *reinterpret_cast<float*>(dl + o) = x - h;
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads32, 1)
    fwd_f32_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, float* __restrict__ O, float* __restrict__ LSE, int BH,
                   int M, int N, float scale_log2_signed, int parts, float* __restrict__ ws,
                   unsigned long long* __restrict__ counters, uint32_t epoch, DevStatus* status,
                   unsigned long long budget_ns) {
  extern __shared__ uint8_t smem_raw[];
  F32Hdr* hdr = reinterpret_cast<F32Hdr*>(smem_raw);
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t data = (raw + 1024u + 1023u) & ~1023u;
  const uint32_t sQh = data, sQl = data + kQBytes;
  auto sKh = [&](int st) { return data + 2 * kQBytes + st * 5 * kKBytes; };
  auto sKl = [&](int st) { return sKh(st) + kKBytes; };
  auto sV = [&](int st) { return sKh(st) + 2 * kKBytes; };
  auto sVth = [&](int st) { return sKh(st) + 3 * kKBytes; };
  auto sVtl = [&](int st) { return sKh(st) + 4 * kKBytes; };
  auto gen = [&](uint32_t a) { return reinterpret_cast<float4*>(smem_raw + (a - raw)); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (M + kBM32 - 1) / kBM32;
  const int nkb = (N + kBN32 - 1) / kBN32;
  const int tiles = BH * nqt;
  // scale < 0: the score product is negated in the tensor core and the softmax scales by |scale|.
  // |scale| is kept above 1e-30 so that a masked score (-inf) times it stays -inf when scale = 0
  // (every visible weight is then exp2 of about 0, i.e. 1).
  const bool neg_scale = scale_log2_signed < 0.f;
  const float scale_log2 = fmaxf(fabsf(scale_log2_signed), 1e-30f);

  // Unit w = (tile w / parts, part w % parts): the tile's key blocks [jb, jb + nb) of its part.
  // With parts > 1 each part leaves an unnormalised partial and counts itself in on its tile;
  // the part that counts in last merges the others into its own and writes O and LSE (no CTA
  // waits for another). Empty parts (causal tiles with fewer blocks than parts) are skipped by
  // every role.
  const int units = tiles * parts;
  auto tile_of = [&](int w, int& bh, int& q0, int& jb, int& nb) {
    const int tile = w / parts, part = w - tile * parts;
    const int qt_rev = tile / BH;
    bh = tile - qt_rev * BH;
    const int qt = CAUSAL ? nqt - 1 - qt_rev : qt_rev;  // causal: heaviest tiles first
    q0 = qt * kBM32;
    const int nbt = CAUSAL ? min(nkb, (q0 + kBM32 - 1) / kBN32 + 1) : nkb;
    jb = part * nbt / parts;
    nb = (part + 1) * nbt / parts - jb;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&hdr->q_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->q_split), 4);
    ptx::mbar_init(ptx::smem_u32(&hdr->q_empty), 1);
    for (int s = 0; s < kStages32; ++s) {
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_split[s]), 4);
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->p_full), 4);
    ptx::mbar_init(ptx::smem_u32(&hdr->o_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMma32) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernFwdF32};
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProd32) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      int n = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
        int bh, q0, jb, nb;
        tile_of(w, bh, q0, jb, nb);
        if (nb == 0) continue;
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->q_empty), (n & 1) ^ 1, wc, 10)) break;
        ++n;
        const uint32_t qf = ptx::smem_u32(&hdr->q_full);
        ptx::mbar_arrive_expect_tx(qf, kQBytes);
        for (int c = 0; c < 2; ++c) ptx::tma_load_3d(sQh + c * kQChunk, &tmQ, qf, c * 32, q0, bh);
        for (int j = 0; j < nb; ++j, ++it) {
          const int st = it % kStages32;
          if (!ptx::mbar_wait(ptx::smem_u32(&hdr->kv_empty[st]), ((it / kStages32) & 1u) ^ 1u, wc, 11)) {
            ok = false;
            break;
          }
          const uint32_t f = ptx::smem_u32(&hdr->kv_full[st]);
          ptx::mbar_arrive_expect_tx(f, 2 * kKBytes);
          for (int c = 0; c < 2; ++c) {
            ptx::tma_load_3d(sKh(st) + c * kKChunk, &tmK, f, c * 32, (jb + j) * kBN32, bh);
            ptx::tma_load_3d(sV(st) + c * kKChunk, &tmV, f, c * 32, (jb + j) * kBN32, bh);
          }
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = it > (uint32_t)kStages32 ? it - kStages32 : 0u; k < it; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->kv_full[k % kStages32]), (k / kStages32) & 1u, 100000000ull);
        if (n > 0) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->q_full), static_cast<uint32_t>(n - 1) & 1u, 100000000ull);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ split warps: x -> (tf32 hi, lo)
    const int tid = threadIdx.x - 128;
    uint32_t it = 0;
    int n = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
      int bh, q0, jb, nb;
      tile_of(w, bh, q0, jb, nb);
      if (nb == 0) continue;
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->q_full), n & 1, wc, 40));
      ++n;
      if (!ok) break;
      split_block(gen(sQh), gen(sQl), kQBytes / 16, tid, 128);
      ptx::fence_proxy_async_smem();  // generic stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->q_split));
      for (int j = 0; j < nb; ++j, ++it) {
        const int st = it % kStages32;
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->kv_full[st]), (it / kStages32) & 1u, wc, 41));
        if (!ok) break;
        split_block(gen(sKh(st)), gen(sKl(st)), kKBytes / 16, tid, 128);
        split_transpose_v(reinterpret_cast<const float*>(gen(sV(st))), reinterpret_cast<float*>(gen(sVth(st))),
                          reinterpret_cast<float*>(gen(sVtl(st))), tid, 128);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->kv_split[st]));
      }
    }
  } else if (warp == kWarpMma32) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id =
          ptx::idesc_f32acc(kBM32, kBN32, ptx::kFmtTF32, ptx::kFmtTF32, false, false) | (neg_scale ? ptx::kNegateA : 0u);
      constexpr uint32_t id_pv = ptx::idesc_f32acc(kBM32, kD32, ptx::kFmtTF32, ptx::kFmtTF32, false, false);
      uint32_t it = 0, p_ph = 0;
      int n = 0;
      bool ok = true;
      // K-major operand with 32-column chunks of `chunk` bytes: k-step ks covers 8 columns
      auto kdesc = [](uint32_t base, uint32_t chunk, int ks) {
        return ptx::sdesc_sw128(base + (ks >> 2) * chunk + (ks & 3) * 32, 16, 1024);
      };
      for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
        int bh, q0, jb, nb;
        tile_of(w, bh, q0, jb, nb);
        if (nb == 0) continue;
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->q_split), n & 1, wc, 20)) break;
        ++n;
        ptx::tc_fence_after();
        for (int j = 0; j < nb; ++j, ++it) {
          const int st = it % kStages32;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->kv_split[st]), (it / kStages32) & 1u, wc, 21);
          if (!ok) break;
          ptx::tc_fence_after();
          // S = Qh Kh^T + Ql Kh^T + Qh Kl^T  (S/P_hi region must be free: the previous
          // P V, issued earlier by this thread, has read P_hi)
#pragma unroll
          for (int ks = 0; ks < kD32 / 8; ++ks) {
            ptx::mma_tf32_ss(tmem, kdesc(sQh, kQChunk, ks), kdesc(sKh(st), kKChunk, ks), id, ks > 0);
            ptx::mma_tf32_ss(tmem, kdesc(sQl, kQChunk, ks), kdesc(sKh(st), kKChunk, ks), id, 1);
            ptx::mma_tf32_ss(tmem, kdesc(sQh, kQChunk, ks), kdesc(sKl(st), kKChunk, ks), id, 1);
          }
          ptx::tc_commit(ptx::smem_u32(&hdr->s_full));
          if (j == nb - 1) ptx::tc_commit(ptx::smem_u32(&hdr->q_empty));
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->p_full), p_ph, wc, 22);
          if (!ok) break;
          p_ph ^= 1u;
          ptx::tc_fence_after();
          // O_j = Ph Vh + Pl Vh + Ph Vl with V^T K-major: 8 keys per k-step; each block
          // starts from zero and the softmax threads add the partials in f32 registers
#pragma unroll
          for (int ks = 0; ks < kBN32 / 8; ++ks) {
            const uint64_t vh = kdesc(sVth(st), kKChunk, ks);
            const uint64_t vl = kdesc(sVtl(st), kKChunk, ks);
            ptx::mma_tf32_ts(tmem + 128, tmem + 0 + ks * 8, vh, id_pv, ks > 0);
            ptx::mma_tf32_ts(tmem + 128, tmem + 64 + ks * 8, vh, id_pv, 1);
            ptx::mma_tf32_ts(tmem + 128, tmem + 0 + ks * 8, vl, id_pv, 1);
          }
          ptx::tc_commit(ptx::smem_u32(&hdr->kv_empty[st]));
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&hdr->o_full));
      }
      ptx::tc_commit(ptx::smem_u32(&hdr->mma_done));
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done), 0u, 1000000000ull);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax / epilogue (one row per thread)
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_sel, tPl = tmem + 64 + lane_sel, tO = tmem + 128 + lane_sel;
    uint32_t s_ph = 0;
    int n = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
      int bh, q0, jb, nb;
      tile_of(w, bh, q0, jb, nb);
      if (nb == 0) continue;
      const int row = q0 + warp * 32 + lane;
      float m2 = -INFINITY, l = 0.f;
      float oacc[kD32];
#pragma unroll
      for (int i = 0; i < kD32; ++i) oacc[i] = 0.f;
      // adds the finished block partial P V (scaled to the current max) into oacc
      auto add_partial = [&]() {
#pragma unroll
        for (int c = 0; c < kD32; c += 32) {
          uint32_t t[32];
          ptx::tmem_ld32(tO + c, t);
          ptx::tmem_wait_ld32(t);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 a = ptx::fadd2(make_float2(oacc[c + i], oacc[c + i + 1]),
                                        make_float2(__uint_as_float(t[i]), __uint_as_float(t[i + 1])));
            oacc[c + i] = a.x;
            oacc[c + i + 1] = a.y;
          }
        }
      };
      for (int j = 0; j < nb; ++j) {
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->s_full), s_ph, wc, 30));
        if (!ok) break;
        s_ph ^= 1u;
        ptx::tc_fence_after();
        // S(j) complete implies P V of block j-1 complete (issued before it by the same thread)
        if (j > 0) add_partial();
        const int k0 = (jb + j) * kBN32;
        const bool edge = k0 + kBN32 > N || (CAUSAL && k0 + kBN32 - 1 > q0);
        auto load_s = [&](int c, uint32_t* r) {
          ptx::tmem_ld32(tS + c, r);
          ptx::tmem_wait_ld32(r);
          if (edge) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int key = k0 + c + i;
              if (key >= N || (CAUSAL && key > row)) r[i] = __float_as_uint(-INFINITY);
            }
          }
        };
        // the block maximum in four independent chains of three-input max
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN32; c += 32) {
          uint32_t r[32];
          load_s(c, r);
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            mx0 = ptx::fmax3(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
            mx1 = ptx::fmax3(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
            mx2 = ptx::fmax3(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
            mx3 = ptx::fmax3(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
          }
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        const float m_new = fmaxf(m2, mx * scale_log2);
        const float m_safe = m_new == -INFINITY ? 0.f : m_new;
        const float corr = ptx::ex2(m2 - m_safe);  // m2 = -inf on the first block: corr = 0
        if (j > 0 && corr != 1.f) {
#pragma unroll
          for (int i = 0; i < kD32; i += 2) {
            const float2 a = ptx::fmul2(make_float2(oacc[i], oacc[i + 1]), make_float2(corr, corr));
            oacc[i] = a.x;
            oacc[i + 1] = a.y;
          }
        }
        m2 = m_new;
        // P = 2^(s c - m) by pairs on the f32x2 pipe, its sum in two independent chains, and its
        // split into the tf32 hi part and the remainder
        const float2 c2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m_safe, -m_safe);
        float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kBN32; c += 32) {
          uint32_t r[32], plo[32];
          load_s(c, r);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = ptx::ffma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
            const float2 p = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            if (i & 2)
              sum_b = ptx::fadd2(sum_b, p);
            else
              sum_a = ptx::fadd2(sum_a, p);
            const float2 h = make_float2(tf32_hi(p.x), tf32_hi(p.y));
            const float2 lo = ptx::fsub2(p, h);
            r[i] = __float_as_uint(h.x);
            r[i + 1] = __float_as_uint(h.y);
            plo[i] = __float_as_uint(lo.x);
            plo[i + 1] = __float_as_uint(lo.y);
          }
          ptx::tmem_st32(tS + c, r);
          ptx::tmem_st32(tPl + c, plo);
        }
        const float2 sum2 = ptx::fadd2(sum_a, sum_b);
        l = fmaf(l, corr, sum2.x + sum2.y);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->p_full));
      }
      if (!ok) break;
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->o_full), n & 1, wc, 31));
      if (!ok) break;
      ++n;
      ptx::tc_fence_after();
      add_partial();
      if (parts > 1) {
        // unnormalised partial of this part, column-major (a warp's 32 rows of a column are
        // one contiguous line): O [64][128], m [128], l [128]
        const int tile = w / parts, part = w - tile * parts;
        const int nbt = CAUSAL ? min(nkb, (q0 + kBM32 - 1) / kBN32 + 1) : nkb;
        auto nonempty = [&](int p) { return (p + 1) * nbt / parts > p * nbt / parts; };
        auto slot_of = [&](int p) { return ws + (static_cast<size_t>(tile) * parts + p) * kF32Slot; };
        const int r = warp * 32 + lane;
        float* slot = slot_of(part);
#pragma unroll
        for (int c = 0; c < kD32; ++c) __stcg(slot + c * kBM32 + r, oacc[c]);
        __stcg(slot + kD32 * kBM32 + r, m2);
        __stcg(slot + kD32 * kBM32 + kBM32 + r, l);
        ptx::tc_fence_before();
        __threadfence();  // every lane's partial, at gpu scope, before the count
        __syncwarp();
        int holders = 0;
        for (int p = 0; p < parts; ++p) holders += nonempty(p) ? 1 : 0;
        // count in on (tile, warp): the 64-bit word holds (epoch << 32) | count, so whatever an
        // earlier launch left there (another epoch) reads as a count of zero
        uint32_t count = 0;
        if (lane == 0) {
          unsigned long long* cw = counters + static_cast<size_t>(tile) * 4 + warp;
          const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
          unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(cw);
          for (uint32_t it = 0; it < (1u << 20); ++it) {
            const unsigned long long nv = (cur >> 32) == epoch ? cur + 1ull : (tag | 1ull);
            const unsigned long long seen = atomicCAS(cw, cur, nv);
            if (seen == cur) {
              count = static_cast<uint32_t>(nv);
              break;
            }
            cur = seen;
          }
          if (count == 0u) ptx::raise_error(wc, kStatusTimeout, 39);
        }
        __syncwarp();  // the other lanes' reads below follow lane 0's count
        count = __shfl_sync(0xFFFFFFFFu, count, 0);
        if (count == 0u) break;
        if (static_cast<int>(count) < holders) continue;  // a later part finishes the tile
        __threadfence();  // the other parts' partials, counted in before this one, are visible
        // merge: m = max_s m_s, weights 2^(m_s - m) (the online-softmax rescaling)
        float mm = m2;
        for (int p = 0; p < parts; ++p)
          if (p != part && nonempty(p)) mm = fmaxf(mm, __ldcg(slot_of(p) + kD32 * kBM32 + r));
        const float a = m2 == -INFINITY ? 0.f : ptx::ex2(m2 - mm);
        l *= a;
#pragma unroll
        for (int c = 0; c < kD32; ++c) oacc[c] *= a;
        for (int p = 0; p < parts; ++p) {
          if (p == part || !nonempty(p)) continue;
          const float* sp = slot_of(p);
          const float mp = __ldcg(sp + kD32 * kBM32 + r);
          const float b = mp == -INFINITY ? 0.f : ptx::ex2(mp - mm);
          l = fmaf(b, __ldcg(sp + kD32 * kBM32 + kBM32 + r), l);
#pragma unroll
          for (int c = 0; c < kD32; ++c) oacc[c] = fmaf(b, __ldcg(sp + c * kBM32 + r), oacc[c]);
        }
        m2 = mm;
      }
      const float inv = 1.f / l;
      const bool valid = row < M;
      const size_t g = static_cast<size_t>(bh) * M + (valid ? row : 0);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(O + g * kD32);
#pragma unroll
        for (int v = 0; v < kD32 / 4; ++v)
          dst[v] = make_float4(oacc[4 * v] * inv, oacc[4 * v + 1] * inv, oacc[4 * v + 2] * inv, oacc[4 * v + 3] * inv);
      }
      if (valid && LSE != nullptr) LSE[g] = (m2 + __log2f(l)) * kLn2_32;
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma32) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
  }
}

template <bool CAUSAL>
cudaError_t launch32(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* O, float* LSE, int BH,
                     int M, int N, float scale, int parts, float* ws, uint32_t epoch, const LaunchCtx& ctx) {
  auto kern = fwd_f32_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem32);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>((M + kBM32 - 1) / kBM32) * BH * parts;
  const int grid = static_cast<int>(units < ctx.num_sms ? units : ctx.num_sms);
  // the tiles' counters follow the partial slots
  unsigned long long* counters =
      parts > 1 ? reinterpret_cast<unsigned long long*>(ws + static_cast<size_t>(units) * kF32Slot) : nullptr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads32);
  cfg.dynamicSmemBytes = kSmem32;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];  // a programmatic dependent of the kernel before it on the stream
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, static_cast<float*>(O), LSE, BH, M, N, scale * kLog2e32, parts, ws,
                            counters, epoch, ctx.status, ctx.wait_budget_ns);
}

}  // namespace

int fwd_f32_parts(int BH, int M, int N, int num_sms) {
  const long long tiles = static_cast<long long>((M + kBM32 - 1) / kBM32) * BH;
  const int nkb = (N + kBN32 - 1) / kBN32;
  if (tiles * 2 > num_sms || nkb < 4) return 1;  // enough tiles, or too few key blocks to share
  long long parts = num_sms / tiles;
  if (parts > nkb / 2) parts = nkb / 2;
  return parts < 2 ? 1 : static_cast<int>(parts);
}

size_t fwd_f32_split_bytes(int BH, int M, int parts) {
  if (parts <= 1) return 0;
  const size_t tiles = static_cast<size_t>((M + kBM32 - 1) / kBM32) * BH;
  // slots, then per tile one counter per softmax warp (4 here, 8 in the pipelined kernel)
  return tiles * parts * kF32Slot * sizeof(float) + tiles * 8 * sizeof(unsigned long long);
}

cudaError_t launch_fwd_f32(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                           int D, float scale, bool causal, int parts, float* ws, uint32_t epoch,
                           const LaunchCtx& ctx) {
  if (D != kD32) return cudaErrorNotSupported;
  if (parts < 1 || (parts > 1 && ws == nullptr)) parts = 1;
  CUtensorMap mq, mk, mv;
  if (!make_tmap_3d(&mq, Q, kF32, D, M, BH, 32, kBM32) || !make_tmap_3d(&mk, K, kF32, D, N, BH, 32, kBN32) ||
      !make_tmap_3d(&mv, V, kF32, D, N, BH, 32, kBN32))
    return cudaErrorInvalidValue;
  return causal ? launch32<true>(mq, mk, mv, O, LSE, BH, M, N, scale, parts, ws, epoch, ctx)
                : launch32<false>(mq, mk, mv, O, LSE, BH, M, N, scale, parts, ws, epoch, ctx);
}

}  // namespace fa
