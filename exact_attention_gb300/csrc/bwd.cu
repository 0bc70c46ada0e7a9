// Backward pass for fp16 / bf16 inputs: delta, then dK/dV, then dQ.
//
// The method is the fused-attention tutorial's backward ("06: Fused attention":
// attn_bwd_delta, attn_bwd_dkdv, attn_bwd_dq): the probabilities are recomputed
// from the stored log-sum-exp, P = exp(scale * q.k - L); delta_i = rowsum(dO o O)
// and dS = P o (dP - delta) ("Flash Attention" notes, "IO complexity");
// dV = P^T dO, dK = scale * dS^T Q, dQ = scale * dS K.
//
// GB300 layout of the work (both gradient kernels): a CTA owns one 128-row tile
// (keys for dK/dV, queries for dQ) and walks the other side in 128-row blocks
// streamed by a TMA producer warp through a two-stage ring; one MMA thread
// issues tcgen05 MMAs with the accumulators in tensor memory; four compute
// warps (one per tensor-memory lane quarter, one tile row per thread) turn the
// two score-like products into packed halves that the next MMAs read straight
// from tensor memory. dK/dV computes the transposed products S^T = K Q^T and
// dP^T = V dO^T so that its rows are keys. P and dS are rounded to the I/O half
// type once, as the MMA operands; everything else accumulates in f32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kT = 128;          // tile rows (keys or queries) and streamed block rows
constexpr int kChunkB = 16384;   // 128 rows x 128 bytes, one swizzled chunk
constexpr int kStagesB = 2;
constexpr int kThreadsB = 192;   // 4 compute warps, producer (4), MMA (5)
constexpr int kWarpProdB = 4;
constexpr int kWarpMmaB = 5;
constexpr float kLog2eB = 1.4426950408889634f;
constexpr int kMinSmem = 120 * 1024;  // keeps one CTA per SM (each allocates all of tensor memory)

// ------------------------------------------------------------------------- delta
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ O, const uint16_t* __restrict__ dO,
                                                        float* __restrict__ delta, long long rows) {
  constexpr int kLPR = D * 2 / 16;          // lanes per row (16-byte vectors)
  constexpr int kRPW = 32 / kLPR;           // rows per warp pass
  const int lane = threadIdx.x & 31;
  const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int sub = lane / kLPR, sl = lane % kLPR;
  for (long long r0 = warp_g * kRPW; r0 < rows; r0 += nwarps * kRPW) {
    const long long r = r0 + sub;
    float acc = 0.f;
    if (r < rows) {
      const uint4 a = *reinterpret_cast<const uint4*>(O + r * D + sl * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(dO + r * D + sl * 8);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = BF16 ? ptx::unpack_bf16x2(wa[i]) : ptx::unpack_f16x2(wa[i]);
        const float2 fb = BF16 ? ptx::unpack_bf16x2(wb[i]) : ptx::unpack_f16x2(wb[i]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int o = kLPR / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (sl == 0 && r < rows) delta[r] = acc;
  }
}

struct BwdHdr {
  unsigned long long fixed_full, fixed_empty;
  unsigned long long full[kStagesB], empty[kStagesB];
  unsigned long long s_full, p_full, acc_full, mma_done;
  uint32_t tmem_base;
  int abort_flag;
  float lse2[kStagesB][kT];   // per streamed block: LSE * log2(e) (dK/dV only)
  float dlt[kStagesB][kT];    // per streamed block: delta (dK/dV only)
};

// the 1024-aligned operand region starts after the header
constexpr uint32_t kHdrBytes = (sizeof(BwdHdr) + 127u) & ~127u;

template <int D>
struct BwdCfg {
  static constexpr int kDC = D / 64;
  static constexpr int kTileBytes = kDC * kChunkB;
  // fixed operands (2 tiles), streamed operands (2 tiles per stage)
  static constexpr int kData = 2 * kTileBytes + kStagesB * 2 * kTileBytes;
  static constexpr int kSmemNeed = 1024 + static_cast<int>(kHdrBytes) + kData;
  static constexpr int kSmem = kSmemNeed > kMinSmem ? kSmemNeed : kMinSmem;
};

// Which part of the work a persistent CTA does next.
struct BwdItem {
  int bh, r0;  // head, first row of this CTA's tile
  int lo, hi;  // streamed blocks [lo, hi)
};

// Scores, in the packed-halves layout an MMA A operand uses in tensor memory.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
}

// K-major 128-row operand at `addr` (D/64 chunks): descriptor for k-step ks.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr, int ks) {
  return ptx::sdesc_sw128(addr + (ks >> 2) * kChunkB + (ks & 3) * 32, 16, 1024);
}
// MN-major operand (rows = reduction dim, D contiguous): descriptor for k-step ks of 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t addr, int ks) {
  return ptx::sdesc_sw128(addr + ks * 2048, kChunkB, 1024);
}

// ---------------------------------------------------------------------- dK / dV
// TMEM: S^T [0,128) -> P^T packed [0,64); dP^T [128,256) -> dS^T packed [128,192);
// dV [256, 256+D); dK [256+D, 256+2D).
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const float* __restrict__ LSE, const float* __restrict__ delta, uint16_t* __restrict__ dK,
                    uint16_t* __restrict__ dV, int BH, int M, int N, float scale, DevStatus* status,
                    unsigned long long budget_ns) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  BwdHdr* hdr = reinterpret_cast<BwdHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kHdrBytes + 1023u) & ~1023u;
  const uint32_t sK = data, sV = data + C::kTileBytes;
  auto sQ = [&](int st) { return data + 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto sdO = [&](int st) { return sQ(st) + C::kTileBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  const int items = BH * nkb;
  const float sl2 = scale * kLog2eB;

  auto item = [&](int w) {
    BwdItem it;
    it.bh = w / nkb;
    const int kb = w - it.bh * nkb;
    it.r0 = kb * kT;
    // causal: query block i has keys <= its last row; start at the block holding query k0
    it.lo = CAUSAL ? min(it.r0 / kT, nqb) : 0;
    it.hi = nqb;
    return it;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 1);
    for (int s = 0; s < kStagesB; ++s) {
      ptx::mbar_init(ptx::smem_u32(&hdr->full[s]), 2);  // TMA bytes + LSE/delta staging
      ptx::mbar_init(ptx::smem_u32(&hdr->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->p_full), 4);
    ptx::mbar_init(ptx::smem_u32(&hdr->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMmaB) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDkDv};

  if (warp == kWarpProdB) {
    // ------------------------------------------------------------ producer (whole warp)
    uint32_t it_s = 0;
    int n_item = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
      const BwdItem itm = item(w);
      if (lane == 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10);
        if (ok) {
          const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
          ptx::mbar_arrive_expect_tx(ff, 2 * C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) {
            ptx::tma_load_3d(sK + c * kChunkB, &tmK, ff, c * 64, itm.r0, itm.bh);
            ptx::tma_load_3d(sV + c * kChunkB, &tmV, ff, c * 64, itm.r0, itm.bh);
          }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      for (int i = itm.lo; i < itm.hi && ok; ++i, ++it_s) {
        const int st = it_s % kStagesB;
        if (lane == 0) ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / kStagesB) & 1u) ^ 1u, wc, 11);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) {
            ptx::tma_load_3d(sQ(st) + c * kChunkB, &tmQ, fb, c * 64, i * kT, itm.bh);
            ptx::tma_load_3d(sdO(st) + c * kChunkB, &tmdO, fb, c * 64, i * kT, itm.bh);
          }
        }
        // LSE (base 2) and delta of the block's queries; past M: P = 0, delta = 0
        for (int q = lane; q < kT; q += 32) {
          const int row = i * kT + q;
          const bool in = row < M;
          const size_t g = static_cast<size_t>(itm.bh) * M + (in ? row : 0);
          hdr->lse2[st][q] = in ? LSE[g] * kLog2eB : INFINITY;
          hdr->dlt[st][q] = in ? delta[g] : 0.f;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fb);
      }
    }
  } else if (warp == kWarpMmaB) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      constexpr uint32_t id_s = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, p_ph = 0;
      int n_item = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
        const BwdItem itm = item(w);
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_full), n_item & 1, wc, 20)) break;
        ptx::tc_fence_after();
        for (int i = itm.lo; i < itm.hi; ++i, ++it_s) {
          const int st = it_s % kStagesB;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), (it_s / kStagesB) & 1u, wc, 21);
          if (!ok) break;
          ptx::tc_fence_after();
          // S^T = K Q^T and dP^T = V dO^T
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            ptx::mma_f16_ss(tmem + 0, kmajor_desc(sK, ks), kmajor_desc(sQ(st), ks), id_s, ks > 0);
            ptx::mma_f16_ss(tmem + 128, kmajor_desc(sV, ks), kmajor_desc(sdO(st), ks), id_s, ks > 0);
          }
          ptx::tc_commit(ptx::smem_u32(&hdr->s_full));
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->p_full), p_ph, wc, 22);
          if (!ok) break;
          p_ph ^= 1u;
          ptx::tc_fence_after();
          // dV += P^T dO, dK += dS^T Q
          const bool acc = i > itm.lo;
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            ptx::mma_f16_ts(tmem + 256, tmem + 0 + ks * 8, mnmajor_desc(sdO(st), ks), id_g, (acc || ks > 0));
            ptx::mma_f16_ts(tmem + 256 + D, tmem + 128 + ks * 8, mnmajor_desc(sQ(st), ks), id_g, (acc || ks > 0));
          }
          ptx::tc_commit(ptx::smem_u32(&hdr->empty[st]));
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&hdr->fixed_empty));
        ptx::tc_commit(ptx::smem_u32(&hdr->acc_full));
      }
      ptx::tc_commit(ptx::smem_u32(&hdr->mma_done));
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps: one key row per thread
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_sel, tdP = tmem + 128 + lane_sel;
    const uint32_t tdV = tmem + 256 + lane_sel, tdK = tmem + 256 + D + lane_sel;
    uint32_t it_s = 0, s_ph = 0;
    int n_item = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
      const BwdItem itm = item(w);
      const int key = itm.r0 + warp * 32 + lane;
      for (int i = itm.lo; i < itm.hi; ++i, ++it_s) {
        const int st = it_s % kStagesB;
        // the stage's LSE/delta are staged before its full barrier completes; the
        // MMAs that read the stage completed before s_full
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->s_full), s_ph, wc, 30) &&
                                         ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), (it_s / kStagesB) & 1u, wc, 31));
        if (!ok) break;
        s_ph ^= 1u;
        ptx::tc_fence_after();
        const float* lse2 = hdr->lse2[st];
        const float* dlt = hdr->dlt[st];
        const int q0 = i * kT;
        const bool diag = CAUSAL && q0 < itm.r0 + kT;  // block may hold queries before this key
#pragma unroll
        for (int c = 0; c < kT; c += 32) {
          uint32_t s[32], dp[32];
          ptx::tmem_ld32(tS + c, s);
          ptx::tmem_ld32(tdP + c, dp);
          ptx::tmem_wait_ld32(s);
          ptx::tmem_wait_ld32(dp);
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float p2[2], d2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int q = c + 2 * k + h;
              float p = ptx::ex2(fmaf(__uint_as_float(s[2 * k + h]), sl2, -lse2[q]));
              if (diag && q0 + q < key) p = 0.f;  // key j is visible to query i iff j <= i
              p2[h] = p;
              d2[h] = p * (__uint_as_float(dp[2 * k + h]) - dlt[q]);
            }
            pp[k] = pack2<BF16>(p2[0], p2[1]);
            pd[k] = pack2<BF16>(d2[0], d2[1]);
          }
          ptx::tmem_st16(tS + c / 2, pp);
          ptx::tmem_st16(tdP + c / 2, pd);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->p_full));
      }
      if (!ok) break;
      // epilogue: dV and scale * dK for this thread's key
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->acc_full), n_item & 1, wc, 32));
      if (!ok) break;
      ptx::tc_fence_after();
      const bool valid = key < N;
      const size_t g = (static_cast<size_t>(itm.bh) * N + (valid ? key : 0)) * D;
      const bool none = itm.lo >= itm.hi;  // no query block: the gradients are zero
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t src = part == 0 ? tdV : tdK;
        uint16_t* dst = part == 0 ? dV : dK;
        const float f = part == 0 ? 1.f : scale;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t a[32];
          ptx::tmem_ld32(src + c, a);
          ptx::tmem_wait_ld32(a);
          uint32_t h[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            h[k] = none ? 0u : pack2<BF16>(__uint_as_float(a[2 * k]) * f, __uint_as_float(a[2 * k + 1]) * f);
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + g + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
          }
        }
      }
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaB) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------------------- dQ
// TMEM: S [0,128) -> dS packed [0,64); dP [128,256); dQ [256, 256+D).
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const float* __restrict__ LSE, const float* __restrict__ delta, uint16_t* __restrict__ dQ, int BH,
                  int M, int N, float scale, DevStatus* status, unsigned long long budget_ns) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  BwdHdr* hdr = reinterpret_cast<BwdHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kHdrBytes + 1023u) & ~1023u;
  const uint32_t sQ = data, sdO = data + C::kTileBytes;
  auto sK = [&](int st) { return data + 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto sV = [&](int st) { return sK(st) + C::kTileBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  const int items = BH * nqb;
  const float sl2 = scale * kLog2eB;

  auto item = [&](int w) {
    BwdItem it;
    // causal: heaviest (last) query blocks first
    const int qb_rev = w / BH;
    it.bh = w - qb_rev * BH;
    const int qb = CAUSAL ? nqb - 1 - qb_rev : qb_rev;
    it.r0 = qb * kT;
    it.lo = 0;
    it.hi = CAUSAL ? min(nkb, (it.r0 + kT - 1) / kT + 1) : nkb;
    return it;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 1);
    for (int s = 0; s < kStagesB; ++s) {
      ptx::mbar_init(ptx::smem_u32(&hdr->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->p_full), 4);
    ptx::mbar_init(ptx::smem_u32(&hdr->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMmaB) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDq};

  if (warp == kWarpProdB) {
    if (lane == 0) {
      uint32_t it_s = 0;
      int n_item = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
        const BwdItem itm = item(w);
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10)) break;
        const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
        ptx::mbar_arrive_expect_tx(ff, 2 * C::kTileBytes);
        for (int c = 0; c < C::kDC; ++c) {
          ptx::tma_load_3d(sQ + c * kChunkB, &tmQ, ff, c * 64, itm.r0, itm.bh);
          ptx::tma_load_3d(sdO + c * kChunkB, &tmdO, ff, c * 64, itm.r0, itm.bh);
        }
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % kStagesB;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / kStagesB) & 1u) ^ 1u, wc, 11);
          if (!ok) break;
          const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) {
            ptx::tma_load_3d(sK(st) + c * kChunkB, &tmK, fb, c * 64, j * kT, itm.bh);
            ptx::tma_load_3d(sV(st) + c * kChunkB, &tmV, fb, c * 64, j * kT, itm.bh);
          }
        }
      }
    }
  } else if (warp == kWarpMmaB) {
    if (lane == 0) {
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      constexpr uint32_t id_s = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, p_ph = 0;
      int n_item = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
        const BwdItem itm = item(w);
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_full), n_item & 1, wc, 20)) break;
        ptx::tc_fence_after();
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % kStagesB;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), (it_s / kStagesB) & 1u, wc, 21);
          if (!ok) break;
          ptx::tc_fence_after();
          // S = Q K^T and dP = dO V^T
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            ptx::mma_f16_ss(tmem + 0, kmajor_desc(sQ, ks), kmajor_desc(sK(st), ks), id_s, ks > 0);
            ptx::mma_f16_ss(tmem + 128, kmajor_desc(sdO, ks), kmajor_desc(sV(st), ks), id_s, ks > 0);
          }
          ptx::tc_commit(ptx::smem_u32(&hdr->s_full));
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->p_full), p_ph, wc, 22);
          if (!ok) break;
          p_ph ^= 1u;
          ptx::tc_fence_after();
          // dQ += dS K
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks)
            ptx::mma_f16_ts(tmem + 256, tmem + 0 + ks * 8, mnmajor_desc(sK(st), ks), id_g, (j > itm.lo || ks > 0));
          ptx::tc_commit(ptx::smem_u32(&hdr->empty[st]));
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&hdr->fixed_empty));
        ptx::tc_commit(ptx::smem_u32(&hdr->acc_full));
      }
      ptx::tc_commit(ptx::smem_u32(&hdr->mma_done));
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps: one query row per thread
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_sel, tdP = tmem + 128 + lane_sel, tdQ = tmem + 256 + lane_sel;
    uint32_t s_ph = 0;
    int n_item = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x, ++n_item) {
      const BwdItem itm = item(w);
      const int row = itm.r0 + warp * 32 + lane;
      const bool valid = row < M;
      const size_t g = static_cast<size_t>(itm.bh) * M + (valid ? row : 0);
      const float lse2 = valid ? LSE[g] * kLog2eB : INFINITY;  // past M: P = 0
      const float dlt = valid ? delta[g] : 0.f;
      for (int j = itm.lo; j < itm.hi; ++j) {
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->s_full), s_ph, wc, 30));
        if (!ok) break;
        s_ph ^= 1u;
        ptx::tc_fence_after();
        const int k0 = j * kT;
        const bool edge = k0 + kT > N || (CAUSAL && k0 + kT - 1 > itm.r0);
#pragma unroll
        for (int c = 0; c < kT; c += 32) {
          uint32_t s[32], dp[32];
          ptx::tmem_ld32(tS + c, s);
          ptx::tmem_ld32(tdP + c, dp);
          ptx::tmem_wait_ld32(s);
          ptx::tmem_wait_ld32(dp);
          uint32_t pd[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float d2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int key = k0 + c + 2 * k + h;
              float p = ptx::ex2(fmaf(__uint_as_float(s[2 * k + h]), sl2, -lse2));
              if (edge && (key >= N || (CAUSAL && key > row))) p = 0.f;
              d2[h] = p * (__uint_as_float(dp[2 * k + h]) - dlt);
            }
            pd[k] = pack2<BF16>(d2[0], d2[1]);
          }
          ptx::tmem_st16(tS + c / 2, pd);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->p_full));
      }
      if (!ok) break;
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->acc_full), n_item & 1, wc, 31));
      if (!ok) break;
      ptx::tc_fence_after();
      const bool none = itm.lo >= itm.hi;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t a[32];
        ptx::tmem_ld32(tdQ + c, a);
        ptx::tmem_wait_ld32(a);
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          h[k] = none ? 0u : pack2<BF16>(__uint_as_float(a[2 * k]) * scale, __uint_as_float(a[2 * k + 1]) * scale);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dQ + g * D + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaB) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_bwd_t(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                         void* dQ, void* dK, void* dV, float* delta, int BH, int M, int N, float scale, int dtype,
                         const LaunchCtx& ctx) {
  using C = BwdCfg<D>;
  // delta = rowsum(dO o O)
  {
    const long long rows = static_cast<long long>(BH) * M;
    const long long warps_needed = (rows + (32 / (D * 2 / 16)) - 1) / (32 / (D * 2 / 16));
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = static_cast<long long>(ctx.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    bwd_delta_kernel<D, BF16><<<static_cast<int>(blocks), 256, 0, ctx.stream>>>(
        static_cast<const uint16_t*>(O), static_cast<const uint16_t*>(dO), delta, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tmap_3d(&mq, Q, dtype, D, M, BH, 64, kT) || !make_tmap_3d(&mk, K, dtype, D, N, BH, 64, kT) ||
      !make_tmap_3d(&mv, V, dtype, D, N, BH, 64, kT) || !make_tmap_3d(&mdo, dO, dtype, D, M, BH, 64, kT))
    return cudaErrorInvalidValue;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  {
    auto kern = bwd_dkdv_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(BH) * nkb;
    const int grid = static_cast<int>(items < ctx.num_sms ? items : ctx.num_sms);
    kern<<<grid, kThreadsB, C::kSmem, ctx.stream>>>(mq, mk, mv, mdo, LSE, delta, static_cast<uint16_t*>(dK),
                                                   static_cast<uint16_t*>(dV), BH, M, N, scale, ctx.status,
                                                   ctx.wait_budget_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = bwd_dq_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(BH) * nqb;
    const int grid = static_cast<int>(items < ctx.num_sms ? items : ctx.num_sms);
    kern<<<grid, kThreadsB, C::kSmem, ctx.stream>>>(mq, mk, mv, mdo, LSE, delta, static_cast<uint16_t*>(dQ), BH, M,
                                                   N, scale, ctx.status, ctx.wait_budget_ns);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, float* delta, int BH, int M, int N, int D, float scale,
                       bool causal, int dtype, const LaunchCtx& ctx) {
  const bool bf = dtype == kBF16;
#define FA_B(DD, BB, CC)                                                                                       \
  if (D == DD && bf == BB && causal == CC)                                                                     \
    return launch_bwd_t<DD, BB, CC>(Q, K, V, O, dO, LSE, dQ, dK, dV, delta, BH, M, N, scale, dtype, ctx);
  FA_B(64, false, false)
  FA_B(64, false, true)
  FA_B(64, true, false)
  FA_B(64, true, true)
  FA_B(128, false, false)
  FA_B(128, false, true)
  FA_B(128, true, false)
  FA_B(128, true, true)
#undef FA_B
  return cudaErrorNotSupported;
}

}  // namespace fa
