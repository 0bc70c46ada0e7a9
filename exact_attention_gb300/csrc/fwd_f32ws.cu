// Forward for f32 inputs (D = 64) with a caller-owned workspace. The method is fwd_f32.cu's
// ("Flash attention, f32": a CTA walks the keys of a 128-row query tile in blocks with a running
// max, denominator and unnormalised accumulator) with another exact split of the f32 products and
// a pipeline that keeps the tensor core busy:
//  * every f32 operand x is split into three bf16 parts, x = x0 + x1 + x2 (x0 = x rounded to bf16,
//    x1 = the remainder rounded, x2 = the last remainder; the subtractions are exact), and
//    A B ~= A0 B0 + A0 B1 + A1 B0 + A0 B2 + A1 B1 + A2 B0 (the dropped terms are about 2^-24
//    relative); six kind::f16 MMAs run faster than the three kind::tf32 ones of fwd_f32.cu, which
//    run at half rate with N = 64;
//  * a prologue kernel splits K and V into their parts once per call, into the workspace, so the
//    main kernel streams ready operands (48 KB per 64-key block) through a four-stage ring;
//  * the softmax warps write the tile's query rows, split, into tensor memory, the A operand of
//    S = Q K^T; eight softmax warps, two per row (32 keys of each block each);
//  * S / P and the block partial of P V are double-buffered in tensor memory, so S(j+1) is computed
//    while the softmax works on block j, and P(j) V(j) while it works on block j+1; one thread
//    issues the score products and another the P V products (one issuing thread reaches only half
//    the tensor core's rate with N = 64 MMAs), the first writing S of a buffer again once P V of
//    the block two back has read P there.
// As in fwd_f32.cu every block's P V starts from zero in tensor memory and the softmax threads add
// the block partials in registers with round-to-nearest adds (the tensor core's f32 accumulation
// truncates). Tensor memory: Q parts at 0, 32, 64 (32 columns each, two bf16 per column); three S
// buffers at 128 + 64 b (64 f32 columns each; P's parts 0 and 1 written over S, part 2 in 32 columns
// of its own), so the score products can run up to three blocks ahead of P V; two block partials of
// O at 384 + 64 o.
// With few query tiles each tile's keys are split over `parts` CTAs. When every CTA holds one such
// part and the parts of a tile can run as one thread-block cluster (parts 2, 4 or 8, all clusters
// resident at once), each part leaves its partial in its own shared memory and, after a cluster
// barrier, each CTA merges 128 / parts rows of the tile from all the parts' shared memory;
// otherwise the partials go through the workspace and the part that counts in last merges them.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBMw = 128;                 // query rows per tile
constexpr int kBNw = 64;                  // keys per block
constexpr int kDw = 64;
constexpr int kPlaneW = kBNw * 128;       // 8 KB: 64 rows of 64 bf16 (128-byte swizzled rows)
constexpr int kStagesW = 4;
constexpr int kStageW = 6 * kPlaneW;      // K parts 0-2, V parts 0-2
constexpr int kThreadsW = 352;            // softmax 0-7, producer 8, MMA issuers 9 (S) and 10 (P V)
constexpr int kWarpProdW = 8, kWarpMmaW = 9, kWarpPvW = 10;
constexpr float kLog2eW = 1.4426950408889634f;
constexpr float kLn2W = 0.6931471805599453f;
constexpr int kPartPitch = kDw + 4;       // cluster merge: a partial's rows in shared memory (floats)
// Tensor memory: Q part p at 32 p; S buffer b (0..2) at 128 + 64 b, P's parts 0 and 1 written over it,
// part 2 at p2_col(b) (96, 320, 352); O partial buffer o (0..1) at 384 + 64 o
constexpr uint32_t cQ = 0, cS = 128, cO = 384;
__device__ __forceinline__ uint32_t p2_col(uint32_t b) { return b == 0u ? 96u : 256u + 32u * (b + 1u); }

struct F32wHdr {
  unsigned long long kv_full[kStagesW], kv_empty[kStagesW];
  unsigned long long q_full;      // the unit's Q rows are in tensor memory (8 softmax warps)
  unsigned long long s_full[3];   // S of buffer b computed
  unsigned long long p_full[3];   // P of buffer b stored (8 warps)
  unsigned long long s_free[3];   // P V has read P of buffer b: S may be computed there again
  unsigned long long pv_done[2];  // P V into O partial buffer o computed
  unsigned long long mma_done[2];
  unsigned long long xchg[4];     // per lane quarter: both softmax warps published their value
  uint32_t tmem_base;
  int abort_flag;
  float xval[3][2][kBMw];         // [block parity, or 2: row sums][half][row]
};
constexpr int kSmemW = 1024 + 4096 + kStagesW * kStageW;
static_assert(sizeof(F32wHdr) <= 4096, "header");
static_assert(kSmemW <= 232448, "shared memory budget");

// (a, b) -> three bf16x2 words w0 + w1 + w2 = (a, b): each word rounds what the earlier ones left
__device__ __forceinline__ void split3(float a, float b, uint32_t& w0, uint32_t& w1, uint32_t& w2) {
  w0 = ptx::pack_bf16x2(a, b);
  const float2 r1 = ptx::fsub2(make_float2(a, b), ptx::unpack_bf16x2(w0));
  w1 = ptx::pack_bf16x2(r1.x, r1.y);
  const float2 r2 = ptx::fsub2(r1, ptx::unpack_bf16x2(w1));
  w2 = ptx::pack_bf16x2(r2.x, r2.y);
}

// K and V [BH][N][64] f32 -> their bf16 parts, three planes each of [BH][N][64] bf16.
__global__ void __launch_bounds__(256) f32_presplit_kernel(const float4* __restrict__ K, const float4* __restrict__ V,
                                                           uint2* __restrict__ kp, uint2* __restrict__ vp,
                                                           long long quads) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // this thread's lines of K and V into L2 while the kernel before finishes (one thread a line;
  // up to 32 MB of them, a quarter of L2)
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < quads && quads <= (1ll << 20);
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    if ((i & 7) == 0) {
      ptx::prefetch_l2(K + i);
      ptx::prefetch_l2(V + i);
    }
  ptx::grid_dep_wait();  // K and V may come from the kernel before this one
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < quads;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 k = K[i], v = V[i];
    uint2 a0, a1, a2, b0, b1, b2;
    split3(k.x, k.y, a0.x, a1.x, a2.x);
    split3(k.z, k.w, a0.y, a1.y, a2.y);
    split3(v.x, v.y, b0.x, b1.x, b2.x);
    split3(v.z, v.w, b0.y, b1.y, b2.y);
    kp[i] = a0;
    kp[i + quads] = a1;
    kp[i + 2 * quads] = a2;
    vp[i] = b0;
    vp[i + quads] = b1;
    vp[i + 2 * quads] = b2;
  }
}

// Cluster merge by the 256 softmax threads of rank r: rows [r R, r R + R) of the tile, R = 128 / P,
// tpr threads a row and cpt columns each, from the partials that the P parts of the tile left in
// their shared memory at `data` (row-major [128][kPartPitch], then m [128] and l [128]; parts
// without keys left none). Every shared::cluster load of a thread is issued before any is used:
// one at a time they cost a round trip each (about 180 ns, measured).
template <int P>
__device__ __forceinline__ void cluster_merge(uint32_t data, int nbt, int q0, int bh, int M, float* __restrict__ O,
                                              float* __restrict__ LSE) {
  constexpr int R = kBMw / P, tpr = 256 / R, cpt = kDw / tpr, nv = cpt / 4;
  const int tid = static_cast<int>(threadIdx.x);
  const int r = static_cast<int>(ptx::cluster_rank()) * R + tid / tpr;
  const int cg = (tid % tpr) * cpt;
  bool has[P];
  uint32_t base[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    has[p] = (p + 1) * nbt / P > p * nbt / P;
    base[p] = ptx::peer_addr(data, static_cast<uint32_t>(p));
  }
  float mp[P], lp[P];
  float4 x[P][nv];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    mp[p] = -INFINITY;
    lp[p] = 0.f;
    if (has[p]) {
      mp[p] = ptx::ld_cluster_f32(base[p] + (kBMw * kPartPitch + r) * 4);
      lp[p] = ptx::ld_cluster_f32(base[p] + (kBMw * kPartPitch + kBMw + r) * 4);
#pragma unroll
      for (int v = 0; v < nv; ++v) x[p][v] = ptx::ld_cluster_v4(base[p] + (r * kPartPitch + cg + 4 * v) * 4);
    }
  }
  float mm = -INFINITY;
#pragma unroll
  for (int p = 0; p < P; ++p) mm = fmaxf(mm, mp[p]);
  float L = 0.f;
  float4 acc[nv];
#pragma unroll
  for (int v = 0; v < nv; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int p = 0; p < P; ++p) {
    if (!has[p] || mp[p] == -INFINITY) continue;
    const float w = ptx::ex2(mp[p] - mm);
    L = fmaf(w, lp[p], L);
#pragma unroll
    for (int v = 0; v < nv; ++v)
      acc[v] = make_float4(fmaf(w, x[p][v].x, acc[v].x), fmaf(w, x[p][v].y, acc[v].y), fmaf(w, x[p][v].z, acc[v].z),
                           fmaf(w, x[p][v].w, acc[v].w));
  }
  const int row = q0 + r;
  if (row < M) {
    const float inv = 1.f / L;
    float4* dst = reinterpret_cast<float4*>(O + (static_cast<size_t>(bh) * M + row) * kDw + cg);
#pragma unroll
    for (int v = 0; v < nv; ++v) dst[v] = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
    if (tid % tpr == 0 && LSE != nullptr) LSE[static_cast<size_t>(bh) * M + row] = (mm + __log2f(L)) * kLn2W;
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreadsW, 1)
    fwd_f32ws_kernel(const __grid_constant__ CUtensorMap tmK0, const __grid_constant__ CUtensorMap tmK1,
                     const __grid_constant__ CUtensorMap tmK2, const __grid_constant__ CUtensorMap tmV0,
                     const __grid_constant__ CUtensorMap tmV1, const __grid_constant__ CUtensorMap tmV2,
                     const float* __restrict__ Q, float* __restrict__ O, float* __restrict__ LSE, int BH, int M, int N,
                     float scale_log2_signed, int parts, int cl, float* __restrict__ ws,
                     unsigned long long* __restrict__ counters, uint32_t epoch, DevStatus* status,
                     unsigned long long budget_ns) {
  extern __shared__ uint8_t smem_raw[];
  F32wHdr* hdr = reinterpret_cast<F32wHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + 4096u + 1023u) & ~1023u;
  auto sK = [&](int st, int part) { return data + st * kStageW + part * kPlaneW; };
  auto sV = [&](int st, int part) { return data + st * kStageW + (3 + part) * kPlaneW; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (M + kBMw - 1) / kBMw;
  const int nkb = (N + kBNw - 1) / kBNw;
  const int tiles = BH * nqt;
  // scale < 0: the score product is negated in the tensor core and the softmax scales by |scale|
  // (kept above 1e-30 so that a masked score times it stays -inf when scale = 0)
  const bool neg_scale = scale_log2_signed < 0.f;
  const float scale_log2 = fmaxf(fabsf(scale_log2_signed), 1e-30f);

  // Unit w = (tile w / parts, part w % parts): the tile's key blocks [jb, jb + nb) of its part
  // (the split and merge of fwd_f32.cu).
  const int units = tiles * parts;
  auto tile_of = [&](int w, int& bh, int& q0, int& jb, int& nb) {
    const int tile = w / parts, part = w - tile * parts;
    const int qt_rev = tile / BH;
    bh = tile - qt_rev * BH;
    const int qt = CAUSAL ? nqt - 1 - qt_rev : qt_rev;  // causal: heaviest tiles first
    q0 = qt * kBMw;
    const int nbt = CAUSAL ? min(nkb, (q0 + kBMw - 1) / kBNw + 1) : nkb;
    jb = part * nbt / parts;
    nb = (part + 1) * nbt / parts - jb;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesW; ++s) {
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->q_full), 8);
    for (int q = 0; q < 4; ++q) ptx::mbar_init(ptx::smem_u32(&hdr->xchg[q]), 2);
    for (int b = 0; b < 3; ++b) {
      ptx::mbar_init(ptx::smem_u32(&hdr->s_full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->p_full[b]), 8);
      ptx::mbar_init(ptx::smem_u32(&hdr->s_free[b]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->pv_done[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->pv_done[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[1]), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMmaW) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  if (warp == kWarpProdW && lane == 0) {
    ptx::prefetch_tmap(&tmK0);
    ptx::prefetch_tmap(&tmK1);
    ptx::prefetch_tmap(&tmK2);
    ptx::prefetch_tmap(&tmV0);
    ptx::prefetch_tmap(&tmV1);
    ptx::prefetch_tmap(&tmV2);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernFwdF32};
  // launched as a programmatic dependent of the prologue: global memory only after it completed,
  // but the softmax warps' first rows of Q (this thread's 128-byte half row) are brought into L2
  // before, while the prologue runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp < 8 && static_cast<int>(blockIdx.x) < tiles * parts) {
    int bh, q0, jb, nb;
    tile_of(static_cast<int>(blockIdx.x), bh, q0, jb, nb);
    const int row = q0 + (warp & 3) * 32 + lane;
    if (nb > 0 && row < M) ptx::prefetch_l2(Q + (static_cast<size_t>(bh) * M + row) * kDw + (warp >> 2) * 32);
  }
  ptx::grid_dep_wait();

  if (warp == kWarpProdW) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      uint32_t g = 0;  // blocks streamed, all units
      bool ok = true;
      for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
        int bh, q0, jb, nb;
        tile_of(w, bh, q0, jb, nb);
        for (int j = 0; j < nb; ++j, ++g) {
          const int st = g % kStagesW;
          if (!ptx::mbar_wait(ptx::smem_u32(&hdr->kv_empty[st]), ((g / kStagesW) & 1u) ^ 1u, wc, 11)) {
            ok = false;
            break;
          }
          const uint32_t f = ptx::smem_u32(&hdr->kv_full[st]);
          ptx::mbar_arrive_expect_tx(f, kStageW);
          const int key0 = (jb + j) * kBNw;
          ptx::tma_load_3d(sK(st, 0), &tmK0, f, 0, key0, bh);
          ptx::tma_load_3d(sK(st, 1), &tmK1, f, 0, key0, bh);
          ptx::tma_load_3d(sK(st, 2), &tmK2, f, 0, key0, bh);
          ptx::tma_load_3d(sV(st, 0), &tmV0, f, 0, key0, bh);
          ptx::tma_load_3d(sV(st, 1), &tmV1, f, 0, key0, bh);
          ptx::tma_load_3d(sV(st, 2), &tmV2, f, 0, key0, bh);
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = g > (uint32_t)kStagesW ? g - kStagesW : 0u; k < g; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->kv_full[k % kStagesW]), (k / kStagesW) & 1u, 100000000ull);
      }
    }
  } else if (warp == kWarpMmaW || warp == kWarpPvW) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    // One thread issues the score products, another the P V products: a thread holds an MMA
    // instruction about 66 cycles whatever its N, so one issuer leaves the N = 64 products at half
    // the tensor core's rate (measured). The score issuer writes S of buffer b again only after
    // P V of the block two back, which read P there, has completed.
    if (lane == 0) {
      const bool scores = warp == kWarpMmaW;
      const uint32_t id_qk =
          ptx::idesc_f32acc(kBMw, kBNw, ptx::kFmtBF16, ptx::kFmtBF16, false, false) | (neg_scale ? ptx::kNegateA : 0u);
      constexpr uint32_t id_pv = ptx::idesc_f32acc(kBMw, kDw, ptx::kFmtBF16, ptx::kFmtBF16, false, true);
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        const bool r = ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
        ptx::tc_fence_after();
        return r;
      };
      // the six products A_x B_y, smallest first, so each k-step adds its largest term last
      constexpr int kPa[6] = {2, 1, 0, 1, 0, 0}, kPb[6] = {0, 1, 2, 0, 1, 0};
      uint32_t g = 0;
      int n = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
        int bh, q0, jb, nb;
        tile_of(w, bh, q0, jb, nb);
        if (nb == 0) continue;
        if (scores) {
          // the unit's Q is in tensor memory (written after the previous unit's last S was read)
          if (!wait(&hdr->q_full, n & 1, 20)) break;
          ++n;
          for (int j = 0; j < nb && ok; ++j) {
            const uint32_t gg = g + j, b = gg % 3u;
            const int st = gg % kStagesW;
            // S_b free: P V of block gg - 3 has read P there; K of block gg landed
            if (gg >= 3) ok = wait(&hdr->s_free[b], ((gg - 3u) / 3u) & 1u, 23);
            if (ok) ok = wait(&hdr->kv_full[st], (gg / kStagesW) & 1u, 21);
            if (!ok) break;
            // S_b = sum of Q_x K_y^T (A from tensor memory, K K-major)
            const uint32_t d = tmem + cS + 64u * b;
#pragma unroll
            for (int ks = 0; ks < kDw / 16; ++ks)
#pragma unroll
              for (int t = 0; t < 6; ++t)
                ptx::mma_f16_ts(d, tmem + cQ + 32 * kPa[t] + ks * 8,
                                ptx::sdesc_sw128(sK(st, kPb[t]) + ks * 32, 16, 1024), id_qk,
                                (ks > 0 || t > 0) ? 1u : 0u);
            ptx::tc_commit(ptx::smem_u32(&hdr->s_full[b]));
          }
        } else {
          for (int j = 0; j < nb && ok; ++j) {
            const uint32_t gg = g + j, b = gg % 3u, ob = gg & 1u;
            const int st = gg % kStagesW;
            // P(gg) stored (the partial two blocks back, which O_ob held, was read before); its S
            // was computed from this stage, so V of block gg has landed too
            ok = wait(&hdr->p_full[b], (gg / 3u) & 1u, 22);
            if (!ok) break;
            // O_ob = sum of P_x V_y for block gg, from zero (V MN-major); then P's buffer and the
            // stage are free
            const uint32_t o = tmem + cO + 64u * ob;
            const uint32_t pcol[3] = {tmem + cS + 64u * b, tmem + cS + 64u * b + 32u, tmem + p2_col(b)};
#pragma unroll
            for (int ks = 0; ks < kBNw / 16; ++ks)
#pragma unroll
              for (int t = 0; t < 6; ++t)
                ptx::mma_f16_ts(o, pcol[kPa[t]] + ks * 8,
                                ptx::sdesc_sw128(sV(st, kPb[t]) + ks * 2048, kPlaneW, 1024), id_pv,
                                (ks > 0 || t > 0) ? 1u : 0u);
            ptx::tc_commit(ptx::smem_u32(&hdr->pv_done[ob]));
            ptx::tc_commit(ptx::smem_u32(&hdr->s_free[b]));
            ptx::tc_commit(ptx::smem_u32(&hdr->kv_empty[st]));
          }
        }
        g += nb;
      }
      const int me = scores ? 0 : 1;
      ptx::tc_commit(ptx::smem_u32(&hdr->mma_done[me]));
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[me]), 0u, 1000000000ull);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    // Two warps per tensor-memory lane quarter: warp (quarter, half) takes keys [32 half, +32) of
    // each block for its 32 rows and D columns [32 half, +32) of O (and of Q). The halves of a
    // row exchange their block maxima (and, at the end, their sums) through shared memory and a
    // two-arrival barrier per quarter.
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(half * 32);
    const int rr = quarter * 32 + lane;  // row within the tile
    const uint32_t xbar = ptx::smem_u32(&hdr->xchg[quarter]);
    uint32_t g = 0, nx = 0;  // blocks processed; exchanges done on xbar
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    // publishes this lane's value in slot (p, half) and returns the other half's from (p, 1 - half)
    auto exchange = [&](int p, float v, float& other) {
      hdr->xval[p][half][rr] = v;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(xbar);
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(xbar, (nx++) & 1u, wc, 35));
      other = hdr->xval[p][1 - half][rr];
      return r;
    };
    for (int w = blockIdx.x; w < units && ok; w += gridDim.x) {
      int bh, q0, jb, nb;
      tile_of(w, bh, q0, jb, nb);
      if (nb == 0) continue;
      const int row = q0 + rr;
      // this half of the row of Q, split into its three bf16 parts, into tensor memory (rows past
      // M: zeros); part p's 16 columns of this half at 32 p + 16 half
      {
        const float4* qrow =
            reinterpret_cast<const float4*>(Q + (static_cast<size_t>(bh) * M + (row < M ? row : 0)) * kDw + c0);
        uint32_t w0[16], w1[16], w2[16];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 x = row < M ? qrow[v] : make_float4(0.f, 0.f, 0.f, 0.f);
          split3(x.x, x.y, w0[2 * v], w1[2 * v], w2[2 * v]);
          split3(x.z, x.w, w0[2 * v + 1], w1[2 * v + 1], w2[2 * v + 1]);
        }
        ptx::tmem_st16(tmem + lane_sel + cQ + c0 / 2, w0);
        ptx::tmem_st16(tmem + lane_sel + cQ + 32 + c0 / 2, w1);
        ptx::tmem_st16(tmem + lane_sel + cQ + 64 + c0 / 2, w2);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->q_full));
      }
      float m2 = -INFINITY, l = 0.f;  // l: this half's share of the row sum
      float oacc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) oacc[i] = 0.f;
      // this warp's 32 columns of the block partial of buffer b
      auto load_partial = [&](uint32_t b, uint32_t* t) {
        ptx::tmem_ld32(tmem + lane_sel + cO + 64u * b + c0, t);
        ptx::tmem_wait_ld32(t);
      };
      for (int j = 0; j < nb; ++j) {
        const uint32_t gg = g + j, b = gg % 3u, ob = gg & 1u;
        ok = wait_all(&hdr->s_full[b], (gg / 3u) & 1u, 30);
        if (!ok) break;
        const uint32_t tB = tmem + lane_sel + cS + 64u * b;  // this lane quarter's rows of buffer b
        const int k0 = (jb + j) * kBNw + static_cast<int>(c0);  // first key of this warp's columns
        const bool edge = k0 + 32 > N || (CAUSAL && k0 + 31 > q0);
        uint32_t r[32];
        ptx::tmem_ld32(tB + c0, r);
        ptx::tmem_wait_ld32(r);
        if (edge) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = k0 + i;
            if (key >= N || (CAUSAL && key > row)) r[i] = __float_as_uint(-INFINITY);
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          mx0 = ptx::fmax3(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
          mx1 = ptx::fmax3(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
          mx2 = ptx::fmax3(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
          mx3 = ptx::fmax3(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
        }
        float mo;
        ok = exchange(static_cast<int>(gg & 1u), fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)), mo);
        if (!ok) break;
        const float mx = fmaxf(fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)), mo);
        const float m_new = fmaxf(m2, mx * scale_log2);
        const float m_safe = m_new == -INFINITY ? 0.f : m_new;
        const float corr = ptx::ex2(m2 - m_safe);  // m2 = -inf on the first block: corr = 0
        // P = 2^(s c - m) by pairs, its sum in two chains, split into its three bf16 parts; parts 0
        // and 1 go over S (both halves have read their S: they passed the exchange), part 2 beside it
        const float2 c2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m_safe, -m_safe);
        float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
        uint32_t w0[16], w1[16], w2[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = ptx::ffma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
          const float2 p = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
          if (i & 2)
            sum_b = ptx::fadd2(sum_b, p);
          else
            sum_a = ptx::fadd2(sum_a, p);
          split3(p.x, p.y, w0[i / 2], w1[i / 2], w2[i / 2]);
        }
        ptx::tmem_st16(tB + c0 / 2, w0);
        ptx::tmem_st16(tB + 32 + c0 / 2, w1);
        ptx::tmem_st16(tmem + lane_sel + p2_col(b) + c0 / 2, w2);
        // P(gg) stored: its P V may run at once. The O partial buffer it writes held block gg - 2's
        // partial, which this warp read during the previous block, so the hand-over does not wait
        // for block gg - 1's P V, read next.
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->p_full[b]));
        const float2 sum2 = ptx::fadd2(sum_a, sum_b);
        // the previous block's partial joins the accumulator; both go to the new maximum
        if (j > 0) {
          ok = wait_all(&hdr->pv_done[ob ^ 1u], ((gg - 1u) >> 1) & 1u, 32);
          if (!ok) break;
          uint32_t t[32];
          load_partial(ob ^ 1u, t);
          const float2 cc = make_float2(corr, corr);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 a = ptx::fadd2(make_float2(oacc[i], oacc[i + 1]),
                                        make_float2(__uint_as_float(t[i]), __uint_as_float(t[i + 1])));
            const float2 sc = corr != 1.f ? ptx::fmul2(a, cc) : a;
            oacc[i] = sc.x;
            oacc[i + 1] = sc.y;
          }
        }
        l = fmaf(l, corr, sum2.x + sum2.y);
        m2 = m_new;
      }
      if (!ok) break;
      {
        const uint32_t gl = g + nb - 1;
        ok = wait_all(&hdr->pv_done[gl & 1u], (gl >> 1) & 1u, 31);
        if (!ok) break;
        uint32_t t[32];
        load_partial(gl & 1u, t);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 a = ptx::fadd2(make_float2(oacc[i], oacc[i + 1]),
                                      make_float2(__uint_as_float(t[i]), __uint_as_float(t[i + 1])));
          oacc[i] = a.x;
          oacc[i + 1] = a.y;
        }
      }
      g += nb;
      // the row's sum: this half's plus the other's (slot 2)
      {
        float lo;
        ok = exchange(2, l, lo);
        if (!ok) break;
        l += lo;
      }
      if (cl) {
        // this part's partial into this CTA's shared memory, row-major [128][kPartPitch], then m
        // and l; merged after the cluster barrier below. The K/V stages are free: every block's
        // copies have landed and the products that read them have completed.
        float* sp = reinterpret_cast<float*>(smem_raw + (data - ptx::smem_u32(smem_raw)));
        float4* dst = reinterpret_cast<float4*>(sp + rr * kPartPitch + c0);
#pragma unroll
        for (int v = 0; v < 8; ++v) dst[v] = make_float4(oacc[4 * v], oacc[4 * v + 1], oacc[4 * v + 2], oacc[4 * v + 3]);
        if (half == 0) {
          sp[kBMw * kPartPitch + rr] = m2;
          sp[kBMw * kPartPitch + kBMw + rr] = l;
        }
        ptx::tc_fence_before();
        continue;
      }
      if (parts > 1) {
        // unnormalised partial of this part, column-major (a warp's 32 rows of a column are one
        // contiguous line): O [64][128], m [128], l [128] (both halves write the same m and l);
        // counted in per (tile, warp); the part that counts in last on a (tile, warp) merges that
        // warp's columns of the others (m = max, weights 2^(m_s - m)) and writes them
        const int tile = w / parts, part = w - tile * parts;
        const int nbt = CAUSAL ? min(nkb, (q0 + kBMw - 1) / kBNw + 1) : nkb;
        auto nonempty = [&](int p) { return (p + 1) * nbt / parts > p * nbt / parts; };
        auto slot_of = [&](int p) { return ws + (static_cast<size_t>(tile) * parts + p) * kF32SlotFloats; };
        float* slot = slot_of(part);
#pragma unroll
        for (int c = 0; c < 32; ++c) __stcg(slot + (c0 + c) * kBMw + rr, oacc[c]);
        __stcg(slot + kDw * kBMw + rr, m2);
        __stcg(slot + kDw * kBMw + kBMw + rr, l);
        ptx::tc_fence_before();
        __threadfence();  // every lane's partial, at gpu scope, before the count
        __syncwarp();
        int holders = 0;
        for (int p = 0; p < parts; ++p) holders += nonempty(p) ? 1 : 0;
        // the 64-bit word holds (epoch << 32) | count: what an earlier launch left reads as zero
        uint32_t count = 0;
        if (lane == 0) {
          unsigned long long* cw = counters + static_cast<size_t>(tile) * 8 + warp;
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
        __syncwarp();
        count = __shfl_sync(0xFFFFFFFFu, count, 0);
        if (count == 0u) break;
        if (static_cast<int>(count) < holders) continue;  // a later part finishes these columns
        __threadfence();  // the other parts' partials, counted in before this one, are visible
        // (loops unrolled so that several parts' loads are in flight at once: each pass costs a
        // memory round trip per unroll group, not per part)
        float mm = m2;
#pragma unroll 4
        for (int p = 0; p < parts; ++p)
          if (p != part && nonempty(p)) mm = fmaxf(mm, __ldcg(slot_of(p) + kDw * kBMw + rr));
        const float a = m2 == -INFINITY ? 0.f : ptx::ex2(m2 - mm);
        l *= a;
#pragma unroll
        for (int c = 0; c < 32; ++c) oacc[c] *= a;
#pragma unroll 2
        for (int p = 0; p < parts; ++p) {
          if (p == part || !nonempty(p)) continue;
          const float* sp = slot_of(p);
          const float mp = __ldcg(sp + kDw * kBMw + rr);
          const float lp = __ldcg(sp + kDw * kBMw + kBMw + rr);
          float col[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) col[c] = __ldcg(sp + (c0 + c) * kBMw + rr);
          const float bw = mp == -INFINITY ? 0.f : ptx::ex2(mp - mm);
          l = fmaf(bw, lp, l);
#pragma unroll
          for (int c = 0; c < 32; ++c) oacc[c] = fmaf(bw, col[c], oacc[c]);
        }
        m2 = mm;
      }
      const float inv = 1.f / l;
      const bool valid = row < M;
      const size_t gq = static_cast<size_t>(bh) * M + (valid ? row : 0);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(O + gq * kDw + c0);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[v] = make_float4(oacc[4 * v] * inv, oacc[4 * v + 1] * inv, oacc[4 * v + 2] * inv, oacc[4 * v + 3] * inv);
      }
      if (valid && half == 0 && LSE != nullptr) LSE[gq] = (m2 + __log2f(l)) * kLn2W;
      ptx::tc_fence_before();
    }
  }

  if (cl) {
    __syncthreads();      // every warp converged (the .aligned cluster barrier)
    ptx::cluster_sync();  // every part's partial is in its CTA's shared memory
    if (warp < 8) {
      int bh, q0, jb, nb;
      tile_of(blockIdx.x, bh, q0, jb, nb);
      const int nbt = CAUSAL ? min(nkb, (q0 + kBMw - 1) / kBNw + 1) : nkb;
      if (parts == 2)
        cluster_merge<2>(data, nbt, q0, bh, M, O, LSE);
      else if (parts == 4)
        cluster_merge<4>(data, nbt, q0, bh, M, O, LSE);
      else
        cluster_merge<8>(data, nbt, q0, bh, M, O, LSE);
    }
    __syncwarp();
    ptx::cluster_sync();  // the other CTAs have read this one's shared memory
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaW) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t fwd_f32_presplit_bytes(int BH, int N) {
  auto a256 = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
  return 2 * a256(3 * static_cast<size_t>(BH) * N * kDw * 2);  // K's and V's three bf16 planes
}

cudaError_t launch_fwd_f32_presplit(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M,
                                    int N, float scale, bool causal, int parts, float* split_ws, uint32_t epoch,
                                    void* presplit, const LaunchCtx& ctx) {
  if (parts < 1 || (parts > 1 && split_ws == nullptr)) parts = 1;
  auto a256 = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
  const size_t plane = static_cast<size_t>(BH) * N * kDw * 2;  // bytes of one bf16 plane
  char* kp = static_cast<char*>(presplit);
  char* vp = kp + a256(3 * plane);
  CUtensorMap mk[3], mv[3];
  for (int p = 0; p < 3; ++p)
    if (!make_tmap_3d(&mk[p], kp + p * plane, kBF16, kDw, N, BH, 64, kBNw) ||
        !make_tmap_3d(&mv[p], vp + p * plane, kBF16, kDw, N, BH, 64, kBNw))
      return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];  // programmatic dependents of the kernel before each
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  const long long quads = static_cast<long long>(BH) * N * kDw / 4;
  long long pblocks = (quads + 255) / 256;
  if (pblocks > 8ll * ctx.num_sms) pblocks = 8ll * ctx.num_sms;
  cfg.gridDim = dim3(static_cast<unsigned>(pblocks));
  cfg.blockDim = dim3(256);
  cfg.stream = ctx.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, f32_presplit_kernel, static_cast<const float4*>(K),
                                     static_cast<const float4*>(V), reinterpret_cast<uint2*>(kp),
                                     reinterpret_cast<uint2*>(vp), quads);
  if (e != cudaSuccess) return e;
  auto kern = causal ? fwd_f32ws_kernel<true> : fwd_f32ws_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemW);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>((M + kBMw - 1) / kBMw) * BH * parts;
  cfg.gridDim = dim3(static_cast<unsigned>(units < ctx.num_sms ? units : ctx.num_sms));
  cfg.blockDim = dim3(kThreadsW);
  cfg.dynamicSmemBytes = kSmemW;
  // The parts of a tile as one cluster when every CTA holds one part and all the clusters can be
  // resident at once (the hardware places a cluster's CTAs together; a cluster waits only for its
  // own CTAs).
  int cl = 0;
  cudaLaunchAttribute cattr[2];
  cattr[0] = attr[0];
  if ((parts == 2 || parts == 4 || parts == 8) && units <= ctx.num_sms) {
    static int fits[2][9] = {{-1, -1, -1, -1, -1, -1, -1, -1, -1}, {-1, -1, -1, -1, -1, -1, -1, -1, -1}};
    cattr[1].id = cudaLaunchAttributeClusterDimension;
    cattr[1].val.clusterDim.x = static_cast<unsigned>(parts);
    cattr[1].val.clusterDim.y = 1;
    cattr[1].val.clusterDim.z = 1;
    int& f = fits[causal ? 1 : 0][parts];
    if (f < 0) {
      cudaLaunchConfig_t q = cfg;
      q.attrs = cattr;
      q.numAttrs = 2;
      int n = 0;
      f = cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess ? n : 0;
      cudaGetLastError();  // a refused query leaves the split through the workspace
    }
    cl = static_cast<long long>(f) * parts >= units ? 1 : 0;
  }
  if (cl) {
    cfg.attrs = cattr;
    cfg.numAttrs = 2;
  }
  unsigned long long* counters =
      parts > 1 ? reinterpret_cast<unsigned long long*>(split_ws + static_cast<size_t>(units) * kF32SlotFloats)
                : nullptr;
  return cudaLaunchKernelEx(&cfg, kern, mk[0], mk[1], mk[2], mv[0], mv[1], mv[2], static_cast<const float*>(Q),
                            static_cast<float*>(O),
                            LSE, BH, M, N, scale * kLog2eW, parts, cl, split_ws, counters, epoch, ctx.status,
                            ctx.wait_budget_ns);
}

}  // namespace fa
