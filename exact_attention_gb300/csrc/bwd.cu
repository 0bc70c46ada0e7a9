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

#include "bwd_common.cuh"
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

// The CTA's r-th work item of a persistent loop (one CTA per SM): round-robin over the item
// order, every other round reversed when causal (serpentine), so a CTA that took one of the
// heaviest items of a round takes one of the lightest of the next; `items` when none is left.
template <bool CAUSAL>
__device__ __forceinline__ int item_of_round(int r, int items) {
  const int c = (CAUSAL && (r & 1)) ? static_cast<int>(gridDim.x - 1u - blockIdx.x) : static_cast<int>(blockIdx.x);
  const long long w = static_cast<long long>(r) * gridDim.x + c;
  return w < items ? static_cast<int>(w) : items;
}

constexpr int kStagesB = 2;
constexpr int kThreadsB = 192;   // 4 compute warps, producer (4), MMA (5)
constexpr int kWarpProdB = 4;
constexpr int kWarpMmaB = 5;
constexpr int kMinSmem = 120 * 1024;  // keeps one CTA per SM (each allocates all of tensor memory)

// ------------------------------------------------------------------------- delta
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ O, const uint16_t* __restrict__ dO,
                                                        float* __restrict__ delta, float* __restrict__ acc_zero,
                                                        uint32_t* __restrict__ counters_zero, int n_counters,
                                                        long long rows) {
  // launched as a programmatic dependent of the kernel before it on the stream (a previous
  // backward's dQ conversion reads the accumulator this kernel zeroes): wait for it first
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();
  // the fused pass's counters (split schedule) start at zero
  if (blockIdx.x == 0)
    for (int k = threadIdx.x; k < n_counters; k += blockDim.x) counters_zero[k] = 0u;
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
    if (acc_zero != nullptr && r < rows) {  // the row's D f32 of the dQ accumulator start at zero
      float4* z = reinterpret_cast<float4*>(acc_zero + r * D);
#pragma unroll
      for (int k = 0; k < D / 4 / kLPR; ++k) z[sl + k * kLPR] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
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
  // scale < 0: the score product is negated in the tensor core, the exponent scales by |scale|
  // (kept above 1e-30, so that masked scores stay -inf when scale = 0) and dK, dQ take the signed scale
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;

  auto item = [&](int w) {
    BwdItem it;
    // causal: key tiles with the most query blocks (the first ones) go first, all heads of a
    // key tile together; non-causal: the key tiles of a head are adjacent
    int kb;
    if (CAUSAL) {
      kb = w / BH;
      it.bh = w - kb * BH;
    } else {
      it.bh = w / nkb;
      kb = w - it.bh * nkb;
    }
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
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProdB) {
    // ------------------------------------------------------------ producer (whole warp)
    uint32_t it_s = 0, n_fixed = 0;  // n_fixed: K/V loads issued (lane 0)
    int n_item = 0;
    bool ok = true;
    for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
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
          ++n_fixed;
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
    if (lane == 0 && hdr->abort_flag) {  // let issued copies land before shared memory is released
      for (uint32_t k = it_s > (uint32_t)kStagesB ? it_s - kStagesB : 0u; k < it_s; ++k)
        ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % kStagesB]), (k / kStagesB) & 1u, 100000000ull);
      if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
    }
  } else if (warp == kWarpMmaB) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, p_ph = 0;
      int n_item = 0;
      bool ok = true;
      for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
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
            ptx::mma_f16_ss(tmem + 128, kmajor_desc(sV, ks), kmajor_desc(sdO(st), ks), id_dp, ks > 0);
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
        // only items with a query block have accumulators to hand over; an empty item's commit
        // would complete the barrier's next phase too early (two phases ahead of its waiters)
        if (itm.lo < itm.hi) ptx::tc_commit(ptx::smem_u32(&hdr->acc_full));
      }
      ptx::tc_commit(ptx::smem_u32(&hdr->mma_done));
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps: one key row per thread
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_sel, tdP = tmem + 128 + lane_sel;
    const uint32_t tdV = tmem + 256 + lane_sel, tdK = tmem + 256 + D + lane_sel;
    uint32_t it_s = 0, s_ph = 0, n_acc = 0;  // n_acc: items with a query block (acc_full phases)
    int n_item = 0;
    bool ok = true;
    for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
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
      const bool none = itm.lo >= itm.hi;  // no query block: the gradients are zero
      if (!none) {
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&hdr->acc_full), (n_acc++) & 1u, wc, 32));
        if (!ok) break;
      }
      ptx::tc_fence_after();
      const bool valid = key < N;
      const size_t g = (static_cast<size_t>(itm.bh) * N + (valid ? key : 0)) * D;
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

// ------------------------------------------------------- overlapped dK/dV (D = 64) and dQ
// Both keep the scores, dP, the packed MMA operands and the accumulators in
// tensor memory side by side, so the next block's products are computed while
// the compute warps work on this one. Eight compute warps: warp w owns TMEM lane
// quarter w % 4 (one tile row per thread) and the half w / 4 of the streamed
// block's 128 columns. Per block the compute warps signal twice: once the scores
// are read and P is formed (dK/dV: P^T stored), once dP is read and dS stored.
// Two MMA-issuing threads share the work (an MMA instruction holds its issuing
// thread until the tensor pipe accepts it, about the time the pipe's earlier
// work takes, so one issuer left the tensor pipe idle): warp 9 issues the next block's scores at the first signal and its
// dP at the second; warp 10 issues the gradient products of this block at each
// signal and releases the streamed stage (warp 9's products on it completed
// before the compute warps read them). Each barrier's next phase depends on work
// its waiters do after their wait, so no waiter falls two phases behind.
constexpr int kThreadsO = 352;  // compute 0-7, producer 8, MMA issuers 9 (scores) and 10 (gradients)
constexpr int kWarpProdO = 8;
constexpr int kWarpMmaO = 9;
constexpr int kWarpGradO = 10;
constexpr int kStagesMax = 4;

struct OvHdr {
  unsigned long long fixed_full, fixed_empty;
  unsigned long long full[kStagesMax], empty[kStagesMax];
  unsigned long long s_full, dp_full;      // MMA -> compute
  unsigned long long sig1, sig2;           // compute -> MMA (8 warps each)
  unsigned long long s_read;               // compute -> MMA: S^T(i) is in registers (dK/dV, fused)
  unsigned long long free1, free2;         // MMA -> compute: packed operand regions read
  unsigned long long acc_full, mma_done[2];
  // fused dK/dV/dQ only: dQ_i computed, dQ_i read from TMEM, dQ_i staged, staging read by the reduce
  unsigned long long dq_full, dq_free, dq_staged, stg_free;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float nlse2[kStagesMax][kT];  // per streamed block: -LSE * log2(e) (dK/dV only)
  alignas(16) float ndlt[kStagesMax][kT];   // per streamed block: -delta (dK/dV only)
};
constexpr uint32_t kOvHdrBytes = (sizeof(OvHdr) + 127u) & ~127u;

template <int D>
struct OvCfg {
  static constexpr int kDC = D / 64;
  static constexpr int kTileBytes = kDC * kChunkB;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kData = 2 * kTileBytes + kStages * 2 * kTileBytes;
  static constexpr int kSmem = 1024 + static_cast<int>(kOvHdrBytes) + kData;
  static_assert(kSmem <= 232448, "shared memory budget");
};

// The fused dK/dV/dQ kernel (D = 64): K and V, three Q/dO stages, dS^T (32 KB) and the two dQ
// staging boxes (32 KB).
struct FusedCfg {
  static constexpr int kTileBytes = kChunkB;
  static constexpr int kStages = 3;
  static constexpr int kData = 2 * kTileBytes + kStages * 2 * kTileBytes + 2 * kChunkB + 2 * kT * 128;
  static constexpr int kSmem = 1024 + static_cast<int>(kOvHdrBytes) + kData;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kStages <= kStagesMax, "LSE/delta staging");
};

__device__ __forceinline__ void ov_init(OvHdr* hdr, int stages, uint32_t full_count) {
  ptx::mbar_init(ptx::smem_u32(&hdr->fixed_full), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 1);
  for (int st = 0; st < stages; ++st) {
    ptx::mbar_init(ptx::smem_u32(&hdr->full[st]), full_count);
    ptx::mbar_init(ptx::smem_u32(&hdr->empty[st]), 1);
  }
  ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->dp_full), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->sig1), 8);
  ptx::mbar_init(ptx::smem_u32(&hdr->sig2), 8);
  ptx::mbar_init(ptx::smem_u32(&hdr->s_read), 8);
  ptx::mbar_init(ptx::smem_u32(&hdr->free1), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->free2), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->acc_full), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[0]), 1);
  ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[1]), 1);
  hdr->abort_flag = 0;
  ptx::fence_mbar_init();
}

// dK / dV with D = 64. TMEM: S^T [0,128), dP^T [128,256), P^T packed [256,320),
// dS^T packed [320,384), dV [384,448), dK [448,512).
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsO, 1)
    bwd_dkdv64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                      const float* __restrict__ LSE, const float* __restrict__ delta, uint16_t* __restrict__ dK,
                      uint16_t* __restrict__ dV, int BH, int M, int N, float scale, DevStatus* status,
                      unsigned long long budget_ns) {
  constexpr int D = 64;
  using C = OvCfg<D>;
  constexpr uint32_t cS = 0, cdP = 128, cP = 256, cdS = 320, cdV = 384, cdK = 448;
  extern __shared__ uint8_t smem_raw[];
  OvHdr* hdr = reinterpret_cast<OvHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kOvHdrBytes + 1023u) & ~1023u;
  const uint32_t sK = data, sV = data + C::kTileBytes;
  auto sQ = [&](int st) { return data + 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto sdO = [&](int st) { return sQ(st) + C::kTileBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  const int items = BH * nkb;
  // scale < 0: the score product is negated in the tensor core, the exponent scales by |scale|
  // (kept above 1e-30, so that masked scores stay -inf when scale = 0) and dK, dQ take the signed scale
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;
  auto item = [&](int w) {
    BwdItem it;
    // causal: key tiles with the most query blocks (the first ones) go first, all heads of a
    // key tile together; non-causal: the key tiles of a head are adjacent (shared Q/dO in L2)
    int kb;
    if (CAUSAL) {
      kb = w / BH;
      it.bh = w - kb * BH;
    } else {
      it.bh = w / nkb;
      kb = w - it.bh * nkb;
    }
    it.r0 = kb * kT;
    it.lo = CAUSAL ? min(it.r0 / kT, nqb) : 0;  // query blocks before the diagonal see no key here
    it.hi = nqb;
    return it;
  };

  if (threadIdx.x == 0) ov_init(hdr, C::kStages, 2);  // full: TMA bytes + LSE/delta staging
  if (warp == kWarpMmaO) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDkDv};
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProdO) {
    // ------------------------------------------------------------ producer (whole warp)
    // Walks (item, query block) in order. -LSE (base 2) and -delta of a block's queries
    // are read from global memory one block ahead into registers (lane l holds queries
    // l, l+32, l+64, l+96), so their latency overlaps the wait for the next free stage.
    constexpr int kQL = kT / 32;
    float nl_v[kQL], nd_v[kQL];
    auto fetch = [&](const BwdItem& it, int i) {
#pragma unroll
      for (int k = 0; k < kQL; ++k) {
        const int row = i * kT + lane + 32 * k;
        const bool in = row < M;  // past M: P = 0 (exp of -inf), delta = 0
        const size_t g = static_cast<size_t>(it.bh) * M + (in ? row : 0);
        nl_v[k] = in ? -LSE[g] * kLog2eB : -INFINITY;
        nd_v[k] = in ? -delta[g] : 0.f;
      }
    };
    uint32_t it_s = 0, n_fixed = 0;  // n_fixed: K/V loads issued (lane 0)
    int n_item = 0;
    bool ok = true;
    int r = 0;
    int w = item_of_round<CAUSAL>(0, items);
    BwdItem itm{};
    // first item that has a query block (items without one need only their fixed tiles)
    if (w < items) {
      itm = item(w);
      if (itm.lo < itm.hi) fetch(itm, itm.lo);
    }
    for (; w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
      itm = item(w);
      if (lane == 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10);
        if (ok) {
          const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
          ptx::mbar_arrive_expect_tx(ff, 2 * C::kTileBytes);
          ptx::tma_load_3d(sK, &tmK, ff, 0, itm.r0, itm.bh);
          ptx::tma_load_3d(sV, &tmV, ff, 0, itm.r0, itm.bh);
          ++n_fixed;
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      for (int i = itm.lo; i < itm.hi && ok; ++i, ++it_s) {
        const int st = it_s % C::kStages;
        if (lane == 0)
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / C::kStages) & 1u) ^ 1u, wc, 11);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
          ptx::tma_load_3d(sQ(st), &tmQ, fb, 0, i * kT, itm.bh);
          ptx::tma_load_3d(sdO(st), &tmdO, fb, 0, i * kT, itm.bh);
        }
#pragma unroll
        for (int k = 0; k < kQL; ++k) {
          hdr->nlse2[st][lane + 32 * k] = nl_v[k];
          hdr->ndlt[st][lane + 32 * k] = nd_v[k];
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fb);
        // next block's values: this item's next block, else the first block of the next
        // item that has one
        if (i + 1 < itm.hi) {
          fetch(itm, i + 1);
        } else {
          for (int r2 = r + 1, w2 = item_of_round<CAUSAL>(r2, items); w2 < items; w2 = item_of_round<CAUSAL>(++r2, items)) {
            const BwdItem nx = item(w2);
            if (nx.lo < nx.hi) {
              fetch(nx, nx.lo);
              break;
            }
          }
        }
      }
    }
    if (lane == 0 && hdr->abort_flag) {  // let issued copies land before shared memory is released
      for (uint32_t k = it_s > (uint32_t)C::kStages ? it_s - C::kStages : 0u; k < it_s; ++k)
        ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % C::kStages]), (k / C::kStages) & 1u, 100000000ull);
      if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
    }
  } else if (warp == kWarpMmaO || warp == kWarpGradO) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    if (lane == 0) {
      const bool scores = warp == kWarpMmaO;
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, n1 = 0, n2 = 0;
      int n_item = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      auto stage_ready = [&](uint32_t k) { return wait(&hdr->full[k % C::kStages], (k / C::kStages) & 1u, 21); };
      auto qk = [&](uint32_t k) {  // S^T = K Q^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cS, kmajor_desc(sK, ks), kmajor_desc(sQ(st), ks), id_s, ks > 0);
        commit(&hdr->s_full);
      };
      auto vdo = [&](uint32_t k) {  // dP^T = V dO^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cdP, kmajor_desc(sV, ks), kmajor_desc(sdO(st), ks), id_dp, ks > 0);
        commit(&hdr->dp_full);
      };
      for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (scores) {
          if (!wait(&hdr->fixed_full, n_item & 1, 20)) break;
          if (itm.lo < itm.hi) {
            ok = stage_ready(it_s);
            if (!ok) break;
            ptx::tc_fence_after();
            qk(it_s);
            vdo(it_s);
            // the next block's stage has normally landed long ago: check it while the
            // compute warps work, not between their signal and the next scores
            if (itm.lo + 1 < itm.hi && !stage_ready(it_s + 1)) break;
          }
        }
        for (int i = itm.lo; i < itm.hi; ++i, ++it_s) {
          const int st = it_s % C::kStages;
          const bool more = i + 1 < itm.hi;
          const bool acc = i > itm.lo;
          // scores issuer: S^T(i) read (its columns free for S^T(i+1) while the compute warps form
          // P); gradient issuer: P^T(i) stored
          ok = scores ? wait(&hdr->s_read, (n1++) & 1u, 27) : wait(&hdr->sig1, (n1++) & 1u, 22);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) qk(it_s + 1);
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dV += P^T dO
              ptx::mma_f16_ts(tmem + cdV, tmem + cP + ks * 8, mnmajor_desc(sdO(st), ks), id_g, (acc || ks > 0));
            commit(&hdr->free1);
          }
          // dP^T(i) read and dS^T(i) stored
          ok = wait(&hdr->sig2, (n2++) & 1u, 23);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) vdo(it_s + 1);
            if (i + 2 < itm.hi && !stage_ready(it_s + 2)) {
              ok = false;
              break;
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dK += dS^T Q
              ptx::mma_f16_ts(tmem + cdK, tmem + cdS + ks * 8, mnmajor_desc(sQ(st), ks), id_g, (acc || ks > 0));
            commit(&hdr->free2);
            commit(&hdr->empty[st]);
          }
        }
        if (!ok) break;
        // (an item without a query block hands over no accumulators: its commit would complete
        // acc_full's next phase before the compute warps wait for this one)
        if (scores)
          commit(&hdr->fixed_empty);
        else if (itm.lo < itm.hi)
          commit(&hdr->acc_full);
      }
      const int me = scores ? 0 : 1;
      commit(&hdr->mma_done[me]);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[me]), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps: one key row per thread
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(half * 64);  // this warp's query columns [c0, c0 + 64)
    uint32_t it_s = 0, nb = 0;  // blocks processed (all items): s_full/dp_full/free phases
    uint32_t n_acc = 0;         // items with a query block (acc_full phases)
    int n_item = 0;
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    auto signal = [&](unsigned long long* bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(bar));
    };
    for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
      const BwdItem itm = item(w);
      const int key = itm.r0 + quarter * 32 + lane;
      for (int i = itm.lo; i < itm.hi; ++i, ++it_s, ++nb) {
        const int st = it_s % C::kStages;
        // S^T(i) computed; the stage's -LSE/-delta were staged before its full barrier
        ok = wait_all(&hdr->s_full, nb & 1u, 30) &&
             wait_all(&hdr->full[st], (it_s / C::kStages) & 1u, 31);
        if (!ok) break;
        const float* nl = hdr->nlse2[st] + c0;
        const float* nd = hdr->ndlt[st] + c0;
        const int qb = i * kT + static_cast<int>(c0);  // first query of this warp's columns
        const bool diag = CAUSAL && qb < key;          // some of these queries precede the key
        float p[64];
        {
          uint32_t s[64];
          ptx::tmem_ld32(tmem + lane_sel + cS + c0, s);
          ptx::tmem_ld32(tmem + lane_sel + cS + c0 + 32, s + 32);
          ptx::tmem_wait_ld32(s);
          ptx::tmem_wait_ld32(s + 32);
          signal(&hdr->s_read);  // S^T(i+1) may be computed while P is formed
          const float2 c2 = make_float2(sl2, sl2);
#pragma unroll
          for (int q = 0; q < 64; q += 2) {
            const float2 nlq = *reinterpret_cast<const float2*>(nl + q);
            const float2 x = ptx::ffma2(make_float2(__uint_as_float(s[q]), __uint_as_float(s[q + 1])), c2, nlq);
            p[q] = ptx::ex2(x.x);
            p[q + 1] = ptx::ex2(x.y);
            if (diag) {  // key j is visible to query i iff j <= i
              if (qb + q < key) p[q] = 0.f;
              if (qb + q + 1 < key) p[q + 1] = 0.f;
            }
          }
        }
        // P^T(i-1) has been read by dV's MMA before P^T(i) overwrites it
        if (nb > 0) {
          ok = wait_all(&hdr->free1, (nb - 1u) & 1u, 32);
          if (!ok) break;
        }
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = pack2<BF16>(p[c + 2 * k], p[c + 2 * k + 1]);
          ptx::tmem_st16(tmem + lane_sel + cP + (c0 + c) / 2, pk);
        }
        ptx::tmem_wait_st();
        signal(&hdr->sig1);
        // dP^T(i) computed; dS^T = P^T o (dP^T - delta)
        ok = wait_all(&hdr->dp_full, nb & 1u, 33);
        if (ok && nb > 0) ok = wait_all(&hdr->free2, (nb - 1u) & 1u, 34);
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t dp[32];
          ptx::tmem_ld32(tmem + lane_sel + cdP + c0 + c, dp);
          ptx::tmem_wait_ld32(dp);
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 ndq = *reinterpret_cast<const float2*>(nd + c + 2 * k);
            const float2 t = ptx::fadd2(make_float2(__uint_as_float(dp[2 * k]), __uint_as_float(dp[2 * k + 1])), ndq);
            const float2 ds = ptx::fmul2(make_float2(p[c + 2 * k], p[c + 2 * k + 1]), t);
            pk[k] = pack2<BF16>(ds.x, ds.y);
          }
          ptx::tmem_st16(tmem + lane_sel + cdS + (c0 + c) / 2, pk);
        }
        ptx::tmem_wait_st();
        signal(&hdr->sig2);
      }
      if (!ok) break;
      // epilogue: this warp writes columns [32 * half, 32 * half + 32) of dV and scale * dK
      const bool none = itm.lo >= itm.hi;  // no query block: the gradients are zero
      if (!none) {
        ok = wait_all(&hdr->acc_full, (n_acc++) & 1u, 35);
        if (!ok) break;
      }
      const bool valid = key < N;
      const size_t g = (static_cast<size_t>(itm.bh) * N + (valid ? key : 0)) * D + 32 * half;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t a[32];
        ptx::tmem_ld32(tmem + lane_sel + (part == 0 ? cdV : cdK) + 32 * half, a);
        ptx::tmem_wait_ld32(a);
        const float f = part == 0 ? 1.f : scale;
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          h[k] = none ? 0u : pack2<BF16>(__uint_as_float(a[2 * k]) * f, __uint_as_float(a[2 * k + 1]) * f);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>((part == 0 ? dV : dK) + g);
#pragma unroll
          for (int v = 0; v < 4; ++v) d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaO) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Which pieces of work a CTA of the fused pass takes. A piece is an item (key tile of a head)
// with a range of its query blocks.
//  * Classic: whole items, one per round (item_of_round).
//  * Split (non-causal): the contiguous range [c U / G, (c+1) U / G) of the U = items x nqb
//    (item, query block) units, so every CTA streams the same number of blocks and no part-full
//    last round is left. The pieces of an item cut by range boundaries each leave a partial
//    dK / dV; whichever CTA finishes its piece last adds the others in (see the epilogue).
struct FusedPiece {
  BwdItem it;
  int w;     // item index
  int kind;  // 0: the whole item; 1: its first blocks; 2: later blocks (1 and 2: a cut item)
};
template <bool CAUSAL>
struct FusedSched {
  bool split;
  int r;          // classic: next round
  uint32_t u, e;  // split: the remaining unit range
  __device__ static uint32_t start(uint32_t c, uint32_t units) {
    return static_cast<uint32_t>(static_cast<uint64_t>(c) * units / gridDim.x);
  }
  __device__ FusedSched(bool sp, uint32_t units) : split(sp), r(0), u(0), e(0) {
    if (split) {
      u = start(blockIdx.x, units);
      e = start(blockIdx.x + 1, units);
    }
  }
  template <class ItemFn>
  __device__ bool next(FusedPiece& pc, int items, int nqb, const ItemFn& item) {
    if (!split) {
      const int w = item_of_round<CAUSAL>(r, items);
      if (w >= items) return false;
      ++r;
      pc.it = item(w);
      pc.w = w;
      pc.kind = 0;
      return true;
    }
    if (u >= e) return false;
    const int w = static_cast<int>(u / static_cast<uint32_t>(nqb));
    const int i0 = static_cast<int>(u - static_cast<uint32_t>(w) * static_cast<uint32_t>(nqb));
    const uint32_t left = e - u;
    const int i1 = left < static_cast<uint32_t>(nqb - i0) ? i0 + static_cast<int>(left) : nqb;
    pc.it = item(w);
    pc.it.lo = i0;
    pc.it.hi = i1;
    pc.w = w;
    pc.kind = (i0 == 0 && i1 == nqb) ? 0 : (i0 == 0 ? 1 : 2);
    u += static_cast<uint32_t>(i1 - i0);
    return true;
  }
};

// Partial dK / dV of a split item: two slots per CTA (a CTA's range can cut an item at each end),
// each [dV, dK][64 columns][128 key rows] f32 (unscaled); then, per CTA, one counter per compute
// warp for the items whose first block it holds, zeroed by the delta kernel of the call.
constexpr int kFusedSlotFloats = 2 * 64 * kT;

// dK, dV and dQ in one pass over (key tile, query block) with D = 64: the dK/dV kernel above
// with dS^T in shared memory instead of tensor memory. There one buffer serves as the K-major A
// operand of dK += dS^T Q and, read MN-major, as the A operand of dQ_i = dS K (the tutorial's
// dQ kernel recomputes S and dP for that product; here it reuses them). dQ_i lands in the tensor
// memory dS^T had, the compute warps stage it in shared memory as f32 and the drain warp adds it
// into an f32 dQ accumulator in global memory with a bulk tensor reduce (.add; a query block's
// 128 rows of 64 floats are contiguous there). A later kernel scales and converts the
// accumulator. TMEM: S^T [0,128), dP^T [128,256), P^T packed [256,320), dQ_i [320,384),
// dV [384,448), dK [448,512).
// Warps: kCwF compute warps (kCwF / 4 per TMEM lane quarter: each thread takes kQcF of its key
// row's 128 query columns and kDcF of its 64 gradient columns), then the producer, the MMA
// issuers of the scores and of the gradients, and a warp that drains the staging area (the bulk
// reduce-adds of dQ_i and the stores of dV / dK).
constexpr int kCwF = 8;
constexpr int kSlicesF = kCwF / 4;
constexpr int kQcF = kT / kSlicesF;
constexpr int kDcF = 64 / kSlicesF;
constexpr int kWarpProdF = kCwF, kWarpMmaF = kCwF + 1, kWarpGradF = kCwF + 2, kWarpDrainF = kCwF + 3;
constexpr int kThreadsF = (kCwF + 4) * 32;
static_assert(kQcF % 32 == 0 && (kDcF == 16 || kDcF == 32), "compute-warp slicing");
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsF, 1)
    bwd_fused64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const float* __restrict__ LSE, const float* __restrict__ delta,
                       const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                       const __grid_constant__ CUtensorMap tmQacc, int BH, int M, int N,
                       float scale, float* __restrict__ part_ws, uint32_t* __restrict__ counters,
                       uint16_t* __restrict__ dK, uint16_t* __restrict__ dV,
                       DevStatus* status, unsigned long long budget_ns, int inject) {
  constexpr int D = 64;
  using C = FusedCfg;
  constexpr uint32_t cS = 0, cdP = 128, cP = 256, cdQ = 320, cdV = 384, cdK = 448;
  extern __shared__ uint8_t smem_raw[];
  OvHdr* hdr = reinterpret_cast<OvHdr*>(smem_raw);
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t data = (raw + kOvHdrBytes + 1023u) & ~1023u;
  const uint32_t sK = data, sV = data + C::kTileBytes;
  auto sQ = [&](int st) { return data + 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto sdO = [&](int st) { return sQ(st) + C::kTileBytes; };
  // dS^T of the current block: [q chunk 0..1][key 0..127][64 q], 128-byte swizzled rows
  const uint32_t sdS = data + 2 * C::kTileBytes + C::kStages * 2 * C::kTileBytes;
  // dQ_i staged for the reduce: two boxes [32 d][128 queries] f32 in the tensor map's 128-byte
  // swizzled layout (box b holds columns [32 b, 32 b + 32))
  const uint32_t sStg = sdS + 2 * kChunkB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  const int items = BH * nkb;
  // scale < 0: the score product is negated in the tensor core, the exponent scales by |scale|
  // (kept above 1e-30, so that masked scores stay -inf when scale = 0) and dK, dQ take the signed scale
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;
  const bool split = !CAUSAL && part_ws != nullptr;  // the host checks items * nqb < 2^31
  const uint32_t units = split ? static_cast<uint32_t>(items) * static_cast<uint32_t>(nqb) : 0u;
  auto item = [&](int w) {
    BwdItem it;
    // causal: key tiles with the most query blocks (the first ones) go first, all heads of a
    // key tile together; non-causal: the key tiles of a head are adjacent (shared Q/dO in L2)
    int kb;
    if (CAUSAL) {
      kb = w / BH;
      it.bh = w - kb * BH;
    } else {
      it.bh = w / nkb;
      kb = w - it.bh * nkb;
    }
    it.r0 = kb * kT;
    it.lo = CAUSAL ? min(it.r0 / kT, nqb) : 0;  // query blocks before the diagonal see no key here
    it.hi = nqb;
    return it;
  };

  if (threadIdx.x == 0) {
    ov_init(hdr, C::kStages, 2);  // full: TMA bytes + LSE/delta staging
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 2);  // K is read by both issuers here
    ptx::mbar_init(ptx::smem_u32(&hdr->dq_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig1), kCwF);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig2), kCwF);
    ptx::mbar_init(ptx::smem_u32(&hdr->s_read), kCwF);
    ptx::mbar_init(ptx::smem_u32(&hdr->dq_free), kCwF);
    ptx::mbar_init(ptx::smem_u32(&hdr->dq_staged), kCwF);
    ptx::mbar_init(ptx::smem_u32(&hdr->stg_free), 1);
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMmaF) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // launched behind the delta kernel, which also zeroes the dQ accumulator: the set-up above
  // overlaps its tail
  ptx::grid_dep_wait();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDkDv};

  if (warp == kWarpProdF) {
    // ------------------------------------------------------------ producer (whole warp)
    // Walks (item, query block) in order. -LSE (base 2) and -delta of a block's queries
    // are read from global memory one block ahead into registers (lane l holds queries
    // l, l+32, l+64, l+96), so their latency overlaps the wait for the next free stage.
    constexpr int kQL = kT / 32;
    float nl_v[kQL], nd_v[kQL];
    auto fetch = [&](const BwdItem& it, int i) {
#pragma unroll
      for (int k = 0; k < kQL; ++k) {
        const int row = i * kT + lane + 32 * k;
        const bool in = row < M;  // past M: P = 0 (exp of -inf), delta = 0
        const size_t g = static_cast<size_t>(it.bh) * M + (in ? row : 0);
        nl_v[k] = in ? -LSE[g] * kLog2eB : -INFINITY;
        nd_v[k] = in ? -delta[g] : 0.f;
      }
    };
    uint32_t it_s = 0, n_fixed = 0;  // n_fixed: K/V loads issued (lane 0)
    int n_item = 0;
    bool ok = true;
    FusedSched<CAUSAL> sch(split, units);
    FusedPiece pc;
    bool have = sch.next(pc, items, nqb, item);
    // first piece that has a query block (items without one need only their fixed tiles)
    if (have && pc.it.lo < pc.it.hi) fetch(pc.it, pc.it.lo);
    for (; have && ok; have = sch.next(pc, items, nqb, item), ++n_item) {
      const BwdItem itm = pc.it;
      if (lane == 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10);
        if (ok) {
          const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
          ptx::mbar_arrive_expect_tx(ff, 2 * C::kTileBytes);
          ptx::tma_load_3d(sK, &tmK, ff, 0, itm.r0, itm.bh);
          ptx::tma_load_3d(sV, &tmV, ff, 0, itm.r0, itm.bh);
          ++n_fixed;
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      for (int i = itm.lo; i < itm.hi && ok; ++i, ++it_s) {
        const int st = it_s % C::kStages;
        if (lane == 0)
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / C::kStages) & 1u) ^ 1u, wc, 11);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
          ptx::tma_load_3d(sQ(st), &tmQ, fb, 0, i * kT, itm.bh);
          ptx::tma_load_3d(sdO(st), &tmdO, fb, 0, i * kT, itm.bh);
        }
#pragma unroll
        for (int k = 0; k < kQL; ++k) {
          hdr->nlse2[st][lane + 32 * k] = nl_v[k];
          hdr->ndlt[st][lane + 32 * k] = nd_v[k];
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fb);
        // next block's values: this piece's next block, else the first block of the next
        // piece that has one
        if (i + 1 < itm.hi) {
          fetch(itm, i + 1);
        } else {
          FusedSched<CAUSAL> peek = sch;
          FusedPiece nx;
          while (peek.next(nx, items, nqb, item)) {
            if (nx.it.lo < nx.it.hi) {
              fetch(nx.it, nx.it.lo);
              break;
            }
          }
        }
      }
    }
    if (lane == 0 && hdr->abort_flag) {  // let issued copies land before shared memory is released
      for (uint32_t k = it_s > (uint32_t)C::kStages ? it_s - C::kStages : 0u; k < it_s; ++k)
        ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % C::kStages]), (k / C::kStages) & 1u, 100000000ull);
      if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
    }
  } else if (warp == kWarpMmaF || warp == kWarpGradF) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    if (lane == 0) {
      const bool scores = warp == kWarpMmaF;
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      constexpr uint32_t id_q = ptx::idesc_f32acc(kT, D, fmt, fmt, true, true);  // A = dS read MN-major
      uint32_t it_s = 0, n1 = 0, n2 = 0, nq = 0;
      int n_item = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      auto stage_ready = [&](uint32_t k) { return wait(&hdr->full[k % C::kStages], (k / C::kStages) & 1u, 21); };
      auto qk = [&](uint32_t k) {  // S^T = K Q^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cS, kmajor_desc(sK, ks), kmajor_desc(sQ(st), ks), id_s, ks > 0);
        commit(&hdr->s_full);
      };
      auto vdo = [&](uint32_t k) {  // dP^T = V dO^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cdP, kmajor_desc(sV, ks), kmajor_desc(sdO(st), ks), id_dp, ks > 0);
        commit(&hdr->dp_full);
      };
      FusedSched<CAUSAL> sch(split, units);
      FusedPiece pc;
      for (; ok && sch.next(pc, items, nqb, item); ++n_item) {
        const BwdItem itm = pc.it;
        // Both issuers wait for the item's K and V, although only the scores issuer's products
        // need them first: each arrives once per item on fixed_empty, and an issuer that arrived
        // for items without a query block without waiting would run ahead, complete the
        // barrier's phases early and let the producer refill K and V with copies in flight.
        if (!wait(&hdr->fixed_full, n_item & 1, 20)) break;
        if (scores) {
          if (itm.lo < itm.hi) {
            ok = stage_ready(it_s);
            if (!ok) break;
            ptx::tc_fence_after();
            qk(it_s);
            vdo(it_s);
            // the next block's stage has normally landed long ago: check it while the
            // compute warps work, not between their signal and the next scores
            if (itm.lo + 1 < itm.hi && !stage_ready(it_s + 1)) break;
          }
        }
        for (int i = itm.lo; i < itm.hi; ++i, ++it_s) {
          const int st = it_s % C::kStages;
          const bool more = i + 1 < itm.hi;
          const bool acc = i > itm.lo;
          // scores issuer: S^T(i) read (its columns free for S^T(i+1) while the compute warps form
          // P); gradient issuer: P^T(i) stored
          ok = scores ? wait(&hdr->s_read, (n1++) & 1u, 27) : wait(&hdr->sig1, (n1++) & 1u, 22);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) qk(it_s + 1);
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dV += P^T dO
              ptx::mma_f16_ts(tmem + cdV, tmem + cP + ks * 8, mnmajor_desc(sdO(st), ks), id_g, (acc || ks > 0));
            commit(&hdr->free1);
          }
          // dP^T(i) read and dS^T(i) stored
          ok = wait(&hdr->sig2, (n2++) & 1u, 23);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) vdo(it_s + 1);
            if (i + 2 < itm.hi && !stage_ready(it_s + 2)) {
              ok = false;
              break;
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dK += dS^T Q (dS^T K-major in shared memory)
              ptx::mma_f16_ss(tmem + cdK, kmajor_desc(sdS, ks), mnmajor_desc(sQ(st), ks), id_g, (acc || ks > 0));
            // dQ_i = dS K (the same buffer read MN-major: M = queries, K = keys), once the compute
            // warps hold dQ of the previous block
            if (nq > 0 && !wait(&hdr->dq_free, (nq - 1u) & 1u, 26)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)
              ptx::mma_f16_ss(tmem + cdQ, mnmajor_desc(sdS, ks), mnmajor_desc(sK, ks), id_q, ks > 0);
            ++nq;
            commit(&hdr->dq_full);
            commit(&hdr->free2);  // dS^T has been read by both products
            commit(&hdr->empty[st]);
          }
        }
        if (!ok) break;
        // (a piece without a query block hands over no accumulators: its commit would complete
        // acc_full's next phase before the compute warps wait for this one)
        if (!scores && itm.lo < itm.hi) commit(&hdr->acc_full);
        commit(&hdr->fixed_empty);  // K and V read by this thread's products of the item
      }
      const int me = scores ? 0 : 1;
      commit(&hdr->mma_done[me]);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[me]), 0u, 1000000000ull);
    }
  } else if (warp == kWarpDrainF) {
    // ------------------------------------------------------------ staging drain (lane 0)
    // Walks the fills of the staging area in the compute warps' order: per piece, the dQ_i of each
    // of its blocks, then (unless the piece ends in a partial) its dV / dK tiles. Per fill: wait
    // until the eight compute warps have written it, issue the bulk operations, wait until they
    // have read the area and release it for the next fill.
    if (lane == 0) {
      uint32_t ns = 0;
      bool ok = true;
      auto drain = [&](auto&& issue) {
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->dq_staged), ns & 1u, wc, 38)) return false;
        issue();
        ptx::bulk_commit();
        ptx::bulk_wait_read();
        ptx::mbar_arrive(ptx::smem_u32(&hdr->stg_free));
        ++ns;
        return true;
      };
      FusedSched<CAUSAL> sch(split, units);
      FusedPiece pc;
      while (ok && sch.next(pc, items, nqb, item)) {
        const BwdItem itm = pc.it;
        for (int i = itm.lo; i < itm.hi && ok; ++i)
          ok = drain([&] {
            ptx::tma_reduce_add_3d(&tmQacc, sStg, 0, i * kT, itm.bh);
            ptx::tma_reduce_add_3d(&tmQacc, sStg + kT * 128, 32, i * kT, itm.bh);
          });
        if (ok && pc.kind != 2)  // whole items and the first blocks of cut ones store dV / dK
          ok = drain([&] {
            ptx::tma_store_3d(&tmdV, sStg, 0, itm.r0, itm.bh);
            ptx::tma_store_3d(&tmdK, sStg + kChunkB, 0, itm.r0, itm.bh);
          });
      }
      ptx::bulk_wait_all();  // the reduces and stores have completed
    }
  } else {
    // ------------------------------------------------------------ compute warps: one key row per thread
    const int quarter = warp & 3, slice = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(slice * kQcF);  // this warp's query columns [c0, c0 + kQcF)
    const int d0 = slice * kDcF;                              // and gradient columns [d0, d0 + kDcF)
    // kDcF gradient columns of this thread's TMEM lane
    auto ld_grad = [&](uint32_t col, uint32_t* a) {
      if constexpr (kDcF == 32) {
        ptx::tmem_ld32(tmem + lane_sel + col, a);
        ptx::tmem_wait_ld32(a);
      } else {
        ptx::tmem_ld16(tmem + lane_sel + col, a);
        ptx::tmem_wait_ld16(a);
      }
    };
    uint32_t it_s = 0, nb = 0;  // blocks processed (all items): s_full/dp_full/free phases
    uint32_t n_acc = 0;         // pieces with a query block (acc_full phases)
    int n_item = 0;
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    auto signal = [&](unsigned long long* bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(bar));
    };
    // The 32 KB staging area after dS^T is filled by the compute warps and drained by the
    // drain warp's bulk tensor operations: the dQ_i blocks (added into the accumulator) and each
    // piece's dV / dK tiles (stored). A fill first waits until the previous drain has read the
    // area. Warp-uniform result.
    uint32_t nq = 0;  // dQ blocks read back (all items)
    uint32_t ns = 0;  // fills of the staging area
    auto stage = [&](const auto& fill) {
      if (ns > 0 && !wait_all(&hdr->stg_free, (ns - 1u) & 1u, 37)) return false;
      fill();
      ptx::fence_proxy_async_smem();  // staging writes -> the TMA engine
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->dq_staged));
      ++ns;
      return true;
    };
    // dQ_i of the previous block: TMEM -> two f32 boxes [32 d][128 queries] (then the TMEM columns
    // are free for the next product), which the drain warp adds into the accumulator
    auto dq_readout = [&]() {
      if (!wait_all(&hdr->dq_full, nq & 1u, 36)) return false;
      uint32_t a[kDcF];
      ld_grad(cdQ + d0, a);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->dq_free));
      ++nq;
      return stage([&] {
        const int rr = quarter * 32 + lane;  // query row within the block
        // columns [d0, d0 + kDcF) sit in box d0 / 32 from its 16-byte chunk (d0 % 32) / 4
        uint8_t* srow = smem_raw + (sStg - raw) + (d0 / 32) * (kT * 128) + rr * 128;
#pragma unroll
        for (int u = 0; u < kDcF / 4; ++u) {
          const int v = (d0 % 32) / 4 + u;
          *reinterpret_cast<uint4*>(srow + ((v ^ (rr & 7)) << 4)) =
              make_uint4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
        }
      });
    };
    FusedSched<CAUSAL> sch(split, units);
    FusedPiece pc;
    for (; ok && sch.next(pc, items, nqb, item); ++n_item) {
      const BwdItem itm = pc.it;
      const int key = itm.r0 + quarter * 32 + lane;
      for (int i = itm.lo; i < itm.hi; ++i, ++it_s, ++nb) {
        const int st = it_s % C::kStages;
        // S^T(i) computed; the stage's -LSE/-delta were staged before its full barrier
        ok = wait_all(&hdr->s_full, nb & 1u, 30) &&
             wait_all(&hdr->full[st], (it_s / C::kStages) & 1u, 31);
        if (!ok) break;
        const float* nl = hdr->nlse2[st] + c0;
        const float* nd = hdr->ndlt[st] + c0;
        const int qb = i * kT + static_cast<int>(c0);  // first query of this warp's columns
        const bool diag = CAUSAL && qb < key;          // some of these queries precede the key
        float p[kQcF];
        {
          uint32_t s[kQcF];
#pragma unroll
          for (int c = 0; c < kQcF; c += 32) ptx::tmem_ld32(tmem + lane_sel + cS + c0 + c, s + c);
#pragma unroll
          for (int c = 0; c < kQcF; c += 32) ptx::tmem_wait_ld32(s + c);
          signal(&hdr->s_read);  // S^T(i+1) may be computed while P is formed
          const float2 c2 = make_float2(sl2, sl2);
          // the block's -LSE values are read four at a time: every lane reads the same 16 bytes
#pragma unroll
          for (int q = 0; q < kQcF; q += 4) {
            const float4 n4 = *reinterpret_cast<const float4*>(nl + q);
            const float2 x0 = ptx::ffma2(make_float2(__uint_as_float(s[q]), __uint_as_float(s[q + 1])), c2,
                                         make_float2(n4.x, n4.y));
            const float2 x1 = ptx::ffma2(make_float2(__uint_as_float(s[q + 2]), __uint_as_float(s[q + 3])), c2,
                                         make_float2(n4.z, n4.w));
            p[q] = ptx::ex2(x0.x);
            p[q + 1] = ptx::ex2(x0.y);
            p[q + 2] = ptx::ex2(x1.x);
            p[q + 3] = ptx::ex2(x1.y);
            if (diag) {  // key j is visible to query i iff j <= i
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (qb + q + e < key) p[q + e] = 0.f;
            }
          }
        }
        // P^T(i-1) has been read by dV's MMA before P^T(i) overwrites it
        if (nb > 0) {
          ok = wait_all(&hdr->free1, (nb - 1u) & 1u, 32);
          if (!ok) break;
        }
#pragma unroll
        for (int c = 0; c < kQcF; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = pack2<BF16>(p[c + 2 * k], p[c + 2 * k + 1]);
          ptx::tmem_st16(tmem + lane_sel + cP + (c0 + c) / 2, pk);
        }
        ptx::tmem_wait_st();
        signal(&hdr->sig1);
        // dP^T(i) computed; dS^T = P^T o (dP^T - delta)
        ok = wait_all(&hdr->dp_full, nb & 1u, 33);
        if (ok && nb > 0) ok = wait_all(&hdr->free2, (nb - 1u) & 1u, 34);
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < kQcF; c += 32) {
          uint32_t dp[32];
          ptx::tmem_ld32(tmem + lane_sel + cdP + c0 + c, dp);
          ptx::tmem_wait_ld32(dp);
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const float4 n4 = *reinterpret_cast<const float4*>(nd + c + 2 * k);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float2 ndq = e == 0 ? make_float2(n4.x, n4.y) : make_float2(n4.z, n4.w);
              const int kk = k + e;
              const float2 t =
                  ptx::fadd2(make_float2(__uint_as_float(dp[2 * kk]), __uint_as_float(dp[2 * kk + 1])), ndq);
              const float2 ds = ptx::fmul2(make_float2(p[c + 2 * kk], p[c + 2 * kk + 1]), t);
              pk[kk] = pack2<BF16>(ds.x, ds.y);
            }
          }
          // row `key` of dS^T, queries [c0 + c, c0 + c + 32): four 16-byte chunks of the
          // 64-query chunk (c0 + c) / 64
          {
            const int rr = quarter * 32 + lane;
            const int qc = static_cast<int>(c0) + c;
            uint8_t* drow = smem_raw + (sdS - raw) + (qc / 64) * kChunkB + rr * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int v = (qc % 64) / 8 + u;
              *reinterpret_cast<uint4*>(drow + ((v ^ (rr & 7)) << 4)) =
                  make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
          }
        }
        ptx::fence_proxy_async_smem();  // the generic-proxy writes of dS^T -> the tensor core
        signal(&hdr->sig2);
        // dQ of the previous block (its product was issued after the previous sig2)
        if (i > itm.lo) {
          ok = dq_readout();
          if (!ok) break;
        }
      }
      if (ok && itm.lo < itm.hi) ok = dq_readout();  // the piece's last block
      if (!ok) break;
      // epilogue: this warp's columns [d0, d0 + kDcF) of dV and dK, for key row rr
      const bool none = itm.lo >= itm.hi;  // no query block: the gradients are zero
      const int rr = quarter * 32 + lane;
      float g2[2][kDcF];
      if (!none) {
        ok = wait_all(&hdr->acc_full, (n_acc++) & 1u, 35);
        if (!ok) break;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          uint32_t a[kDcF];
          ld_grad((part == 0 ? cdV : cdK) + d0, a);
#pragma unroll
          for (int k = 0; k < kDcF; ++k) g2[part][k] = __uint_as_float(a[k]);
        }
      } else {
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int k = 0; k < kDcF; ++k) g2[part][k] = 0.f;
      }
      ptx::tc_fence_before();
      if (pc.kind != 0) {
        // A piece of a split item. The CTAs holding its later blocks took those pieces first:
        // each writes its raw sums into its slot and counts itself in on the item's counter (one
        // per compute warp, kept for the CTA holding the item's first block). That CTA took its
        // piece last: it waits (bounded) until every other holder has counted in, adds their
        // slots to its own sums and stores dV and dK as a whole item does.
        using S = FusedSched<CAUSAL>;
        const uint32_t u0 = static_cast<uint32_t>(pc.w) * static_cast<uint32_t>(nqb);  // the item's units
        const uint32_t u1 = u0 + static_cast<uint32_t>(nqb);
        // holder of u0 (this branch runs only on the split schedule, where units > 0)
        uint32_t ca = units > 0u ? static_cast<uint32_t>(static_cast<uint64_t>(u0) * gridDim.x / units) : 0u;
        while (ca + 1u < gridDim.x && S::start(ca + 1u, units) <= u0) ++ca;
        while (ca > 0u && S::start(ca, units) > u0) --ca;
        // CTA c's slot for this item: its second (last) one if its range starts before the item
        auto slot_of = [&](uint32_t c) { return 2u * c + (S::start(c, units) < u0 ? 1u : 0u); };
        // slot element (part, column, key row); a warp's 32 rows of one column are one 128-byte line
        auto slot_at = [&](uint32_t sl, int part, int k) {
          return part_ws + static_cast<size_t>(sl) * kFusedSlotFloats + (part * 64 + d0 + k) * kT + rr;
        };
        uint32_t* cnt = counters + static_cast<size_t>(ca) * kCwF + warp;
        if (pc.kind == 2) {
          const uint32_t mine = slot_of(blockIdx.x);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int k = 0; k < kDcF; ++k) __stcg(slot_at(mine, part, k), g2[part][k]);
          __threadfence();  // every lane's slot writes, at gpu scope, before the count
          __syncwarp();
          bool count = true;
          if (inject == kInjectBwdCount) {  // test-only: the lowest CTA starting inside an item never counts in
            uint32_t c = 1u;
            while (c < gridDim.x && S::start(c, units) % static_cast<uint32_t>(nqb) == 0u) ++c;
            count = blockIdx.x != c;
          }
          if (lane == 0 && count) atomicAdd(cnt, 1u);
          continue;
        }
        // the item's first blocks: the other holders' counts, then their slots
        uint32_t others = 0;
        for (uint32_t c = ca + 1u; c < gridDim.x && S::start(c, units) < u1; ++c)
          if (S::start(c + 1u, units) > S::start(c, units)) ++others;
        bool got = true;
        if (lane == 0) {
          const uint64_t t0 = ptx::globaltimer_ns();
          got = false;
          for (uint32_t k = 0; k < (1u << 30); ++k) {
            if (ptx::ld_acquire_u32(cnt) >= others) {
              got = true;
              break;
            }
            if ((k & 255u) == 255u && (*wc.abort_flag || ptx::globaltimer_ns() - t0 > wc.budget_ns)) break;
          }
          if (!got) ptx::raise_error(wc, kStatusTimeout, 39);
        }
        ok = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!ok) break;
        __syncwarp();     // lane 0's acquire, then this barrier, order every lane's slot reads after the writes
        __threadfence();
        for (uint32_t c = ca + 1u; c < gridDim.x && S::start(c, units) < u1; ++c) {
          if (S::start(c + 1u, units) == S::start(c, units)) continue;
          const uint32_t sl = slot_of(c);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int k = 0; k < kDcF; ++k) g2[part][k] += __ldcg(slot_at(sl, part, k));
        }
      }
      // dV and scale * dK in the I/O type, as the two 128 x 64 output tiles (128-byte swizzled
      // rows, the tensor maps' layout; rows past N are clipped by the maps), stored by TMA
      uint32_t hv[kDcF / 2], hk[kDcF / 2];
#pragma unroll
      for (int k = 0; k < kDcF / 2; ++k) {
        hv[k] = none ? 0u : pack2<BF16>(g2[0][2 * k], g2[0][2 * k + 1]);
        hk[k] = none ? 0u : pack2<BF16>(g2[1][2 * k] * scale, g2[1][2 * k + 1] * scale);
      }
      ok = stage([&] {
        uint8_t* row = smem_raw + (sStg - raw) + rr * 128;
#pragma unroll
        for (int u = 0; u < kDcF / 8; ++u) {
          const int v = d0 / 8 + u;  // this warp's 16-byte chunks of the row
          *reinterpret_cast<uint4*>(row + ((v ^ (rr & 7)) << 4)) =
              make_uint4(hv[4 * u], hv[4 * u + 1], hv[4 * u + 2], hv[4 * u + 3]);
          *reinterpret_cast<uint4*>(row + kChunkB + ((v ^ (rr & 7)) << 4)) =
              make_uint4(hk[4 * u], hk[4 * u + 1], hk[4 * u + 2], hk[4 * u + 3]);
        }
      });
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaF) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// dQ. TMEM: S [0,128), dP [128,256), dS packed [256,320), dQ [320, 320+D).
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsO, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const float* __restrict__ LSE, const float* __restrict__ delta, uint16_t* __restrict__ dQ, int BH,
                  int M, int N, float scale, DevStatus* status, unsigned long long budget_ns) {
  using C = OvCfg<D>;
  constexpr uint32_t cS = 0, cdP = 128, cdS = 256, cdQ = 320;
  constexpr int kDH = D / 2;  // dQ columns per warp half in the epilogue
  extern __shared__ uint8_t smem_raw[];
  OvHdr* hdr = reinterpret_cast<OvHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kOvHdrBytes + 1023u) & ~1023u;
  const uint32_t sQ = data, sdO = data + C::kTileBytes;
  auto sK = [&](int st) { return data + 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto sV = [&](int st) { return sK(st) + C::kTileBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  const int items = BH * nqb;
  // scale < 0: the score product is negated in the tensor core, the exponent scales by |scale|
  // (kept above 1e-30, so that masked scores stay -inf when scale = 0) and dK, dQ take the signed scale
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;
  auto item = [&](int w) {
    BwdItem it;
    const int qb_rev = w / BH;  // causal: heaviest (last) query blocks first
    it.bh = w - qb_rev * BH;
    const int qb = CAUSAL ? nqb - 1 - qb_rev : qb_rev;
    it.r0 = qb * kT;
    it.lo = 0;
    it.hi = CAUSAL ? min(nkb, (it.r0 + kT - 1) / kT + 1) : nkb;
    return it;
  };

  if (threadIdx.x == 0) ov_init(hdr, C::kStages, 1);
  if (warp == kWarpMmaO) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDq};
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProdO) {
    if (lane == 0) {
      uint32_t it_s = 0, n_fixed = 0;  // n_fixed: Q/dO loads issued
      int n_item = 0;
      bool ok = true;
      for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10)) break;
        const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
        ptx::mbar_arrive_expect_tx(ff, 2 * C::kTileBytes);
        for (int c = 0; c < C::kDC; ++c) {
          ptx::tma_load_3d(sQ + c * kChunkB, &tmQ, ff, c * 64, itm.r0, itm.bh);
          ptx::tma_load_3d(sdO + c * kChunkB, &tmdO, ff, c * 64, itm.r0, itm.bh);
        }
        ++n_fixed;
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % C::kStages;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / C::kStages) & 1u) ^ 1u, wc, 11);
          if (!ok) break;
          const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) {
            ptx::tma_load_3d(sK(st) + c * kChunkB, &tmK, fb, c * 64, j * kT, itm.bh);
            ptx::tma_load_3d(sV(st) + c * kChunkB, &tmV, fb, c * 64, j * kT, itm.bh);
          }
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = it_s > (uint32_t)C::kStages ? it_s - C::kStages : 0u; k < it_s; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % C::kStages]), (k / C::kStages) & 1u, 100000000ull);
        if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
      }
    }
  } else if (warp == kWarpMmaO || warp == kWarpGradO) {
    // ------------------------------------------------------------ MMA issuers (lane 0)
    if (lane == 0) {
      const bool scores = warp == kWarpMmaO;
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, n1 = 0, n2 = 0;
      int n_item = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      auto stage_ready = [&](uint32_t k) { return wait(&hdr->full[k % C::kStages], (k / C::kStages) & 1u, 21); };
      auto qk = [&](uint32_t k) {  // S = Q K^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cS, kmajor_desc(sQ, ks), kmajor_desc(sK(st), ks), id_s, ks > 0);
        commit(&hdr->s_full);
      };
      auto dov = [&](uint32_t k) {  // dP = dO V^T
        const int st = k % C::kStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss(tmem + cdP, kmajor_desc(sdO, ks), kmajor_desc(sV(st), ks), id_dp, ks > 0);
        commit(&hdr->dp_full);
      };
      for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (scores) {
          if (!wait(&hdr->fixed_full, n_item & 1, 20)) break;
          if (itm.lo < itm.hi) {
            ok = stage_ready(it_s);
            if (!ok) break;
            ptx::tc_fence_after();
            qk(it_s);
            dov(it_s);
            // the next block's stage: checked while the compute warps work
            if (itm.lo + 1 < itm.hi && !stage_ready(it_s + 1)) break;
          }
        }
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % C::kStages;
          const bool more = j + 1 < itm.hi;
          if (scores) {
            // S(j) read
            ok = wait(&hdr->sig1, (n1++) & 1u, 22);
            if (!ok) break;
            ptx::tc_fence_after();
            if (more) qk(it_s + 1);
          }
          // dP(j) read and dS(j) stored
          ok = wait(&hdr->sig2, (n2++) & 1u, 23);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) dov(it_s + 1);
            if (j + 2 < itm.hi && !stage_ready(it_s + 2)) {
              ok = false;
              break;
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dQ += dS K
              ptx::mma_f16_ts(tmem + cdQ, tmem + cdS + ks * 8, mnmajor_desc(sK(st), ks), id_g,
                              (j > itm.lo || ks > 0));
            commit(&hdr->free2);
            commit(&hdr->empty[st]);
          }
        }
        if (!ok) break;
        commit(scores ? &hdr->fixed_empty : &hdr->acc_full);
      }
      const int me = scores ? 0 : 1;
      commit(&hdr->mma_done[me]);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[me]), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps: one query row per thread
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(half * 64);  // this warp's key columns [c0, c0 + 64)
    uint32_t nb = 0;
    int n_item = 0;
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    auto signal = [&](unsigned long long* bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(bar));
    };
    for (int r = 0, w = item_of_round<CAUSAL>(0, items); w < items && ok; w = item_of_round<CAUSAL>(++r, items), ++n_item) {
      const BwdItem itm = item(w);
      const int row = itm.r0 + quarter * 32 + lane;
      const bool valid = row < M;
      const size_t g = static_cast<size_t>(itm.bh) * M + (valid ? row : 0);
      const float nlse2 = valid ? -LSE[g] * kLog2eB : -INFINITY;  // past M: P = 0
      const float ndlt = valid ? -delta[g] : 0.f;
      for (int j = itm.lo; j < itm.hi; ++j, ++nb) {
        ok = wait_all(&hdr->s_full, nb & 1u, 30);
        if (!ok) break;
        const int kb = j * kT + static_cast<int>(c0);  // first key of this warp's columns
        const bool edge = kb + 64 > N || (CAUSAL && kb + 63 > row);
        float p[64];
        {
          uint32_t s[64];
          ptx::tmem_ld32(tmem + lane_sel + cS + c0, s);
          ptx::tmem_ld32(tmem + lane_sel + cS + c0 + 32, s + 32);
          ptx::tmem_wait_ld32(s);
          ptx::tmem_wait_ld32(s + 32);
          const float2 c2 = make_float2(sl2, sl2), nl2 = make_float2(nlse2, nlse2);
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const float2 x = ptx::ffma2(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), c2, nl2);
            p[k] = ptx::ex2(x.x);
            p[k + 1] = ptx::ex2(x.y);
            if (edge) {
              if (kb + k >= N || (CAUSAL && kb + k > row)) p[k] = 0.f;
              if (kb + k + 1 >= N || (CAUSAL && kb + k + 1 > row)) p[k + 1] = 0.f;
            }
          }
        }
        signal(&hdr->sig1);  // S(j) read: the next S may be computed
        ok = wait_all(&hdr->dp_full, nb & 1u, 31);
        if (ok && nb > 0) ok = wait_all(&hdr->free2, (nb - 1u) & 1u, 32);  // dS(j-1) read by dQ's MMA
        if (!ok) break;
        const float2 nd2 = make_float2(ndlt, ndlt);
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t dp[32];
          ptx::tmem_ld32(tmem + lane_sel + cdP + c0 + c, dp);
          ptx::tmem_wait_ld32(dp);
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 t = ptx::fadd2(make_float2(__uint_as_float(dp[2 * k]), __uint_as_float(dp[2 * k + 1])), nd2);
            const float2 ds = ptx::fmul2(make_float2(p[c + 2 * k], p[c + 2 * k + 1]), t);
            pk[k] = pack2<BF16>(ds.x, ds.y);
          }
          ptx::tmem_st16(tmem + lane_sel + cdS + (c0 + c) / 2, pk);
        }
        ptx::tmem_wait_st();
        signal(&hdr->sig2);
      }
      if (!ok) break;
      ok = wait_all(&hdr->acc_full, n_item & 1, 33);
      if (!ok) break;
      const bool none = itm.lo >= itm.hi;
#pragma unroll
      for (int c = 0; c < kDH; c += 32) {
        uint32_t a[32];
        ptx::tmem_ld32(tmem + lane_sel + cdQ + kDH * half + c, a);
        ptx::tmem_wait_ld32(a);
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          h[k] = none ? 0u : pack2<BF16>(__uint_as_float(a[2 * k]) * scale, __uint_as_float(a[2 * k + 1]) * scale);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dQ + g * D + kDH * half + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaO) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// dQ = scale * the f32 accumulator of the fused kernel, rounded to the I/O type.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dQ,
                                                             long long n4, float scale) {
  ptx::grid_dep_wait();  // launched behind the fused kernel
  for (long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * 256) {
    const float4 a = acc[i];
    dQ[i] = make_uint2(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale));
  }
}

// A launch as a programmatic dependent of the kernel before it on the stream (the kernel waits
// with griddepcontrol.wait before touching global memory).
template <class Kern, class... Args>
cudaError_t launch_dependent(Kern kern, int grid, int threads, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_bwd_t(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                         void* dQ, void* dK, void* dV, float* delta, float* dQacc, int BH, int M, int N, float scale,
                         int dtype, const BwdSplit& sp, const LaunchCtx& ctx) {
  using C = BwdCfg<D>;
  const bool split = D == 64 && !CAUSAL && dQacc != nullptr && sp.ws != nullptr;
  uint32_t* counters =
      split ? reinterpret_cast<uint32_t*>(sp.ws + static_cast<size_t>(ctx.num_sms) * 2 * kFusedSlotFloats) : nullptr;
  // delta = rowsum(dO o O)
  {
    const long long rows = static_cast<long long>(BH) * M;
    const long long warps_needed = (rows + (32 / (D * 2 / 16)) - 1) / (32 / (D * 2 / 16));
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = static_cast<long long>(ctx.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    // the fused D = 64 pass accumulates dQ into dQacc, which this kernel zeroes on the way, and
    // its split schedule's counters start at zero
    float* zero = D == 64 ? dQacc : nullptr;
    cudaLaunchConfig_t dcfg{};
    dcfg.gridDim = dim3(static_cast<unsigned>(blocks));
    dcfg.blockDim = dim3(256);
    dcfg.stream = ctx.stream;
    cudaLaunchAttribute dattr[1];
    dattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    dattr[0].val.programmaticStreamSerializationAllowed = 1;
    dcfg.attrs = dattr;
    dcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&dcfg, bwd_delta_kernel<D, BF16>, static_cast<const uint16_t*>(O),
                                       static_cast<const uint16_t*>(dO), delta, zero, counters,
                                       split ? ctx.num_sms * kCwF : 0, rows);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tmap_3d(&mq, Q, dtype, D, M, BH, 64, kT) || !make_tmap_3d(&mk, K, dtype, D, N, BH, 64, kT) ||
      !make_tmap_3d(&mv, V, dtype, D, N, BH, 64, kT) || !make_tmap_3d(&mdo, dO, dtype, D, M, BH, 64, kT))
    return cudaErrorInvalidValue;
  const int nkb = (N + kT - 1) / kT, nqb = (M + kT - 1) / kT;
  if constexpr (D == 64) {
    if (dQacc != nullptr) {  // one pass for dK, dV and dQ (dQ accumulated in f32, then converted)
      const size_t n = static_cast<size_t>(BH) * M * D;
      CUtensorMap macc, mdk, mdv;
      if (!make_tmap_3d(&macc, dQacc, kF32, D, M, BH, 32, kT) || !make_tmap_3d(&mdk, dK, dtype, D, N, BH, 64, kT) ||
          !make_tmap_3d(&mdv, dV, dtype, D, N, BH, 64, kT))
        return cudaErrorInvalidValue;
      const long long items = static_cast<long long>(BH) * nkb;
      auto kern = bwd_fused64_kernel<BF16, CAUSAL>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FusedCfg::kSmem);
      if (e != cudaSuccess) return e;
      // The later kernels are launched as programmatic dependents: each starts its set-up while
      // the kernel before it drains and waits (griddepcontrol.wait) before touching that
      // kernel's results. On the split schedule the CTA holding a cut key tile's first blocks
      // waits (bounded) for the partials of the CTAs holding the rest, which take those pieces
      // first; the launch has one CTA per SM, resident as the SMs free up (as the forward's
      // split schedule relies on).
      cudaLaunchAttribute pdl[1];
      pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      pdl[0].val.programmaticStreamSerializationAllowed = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(split ? ctx.num_sms : (items < ctx.num_sms ? items : ctx.num_sms)));
      cfg.blockDim = dim3(kThreadsF);
      cfg.dynamicSmemBytes = FusedCfg::kSmem;
      cfg.stream = ctx.stream;
      cfg.attrs = pdl;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mdo, LSE, static_cast<const float*>(delta), mdk, mdv, macc, BH,
                             M, N, scale, split ? sp.ws : static_cast<float*>(nullptr), counters,
                             static_cast<uint16_t*>(dK), static_cast<uint16_t*>(dV), ctx.status,
                             ctx.wait_budget_ns, ctx.inject);
      if (e != cudaSuccess) return e;
      const long long n4 = static_cast<long long>(n / 4);
      long long blocks = (n4 + 255) / 256;
      const long long cap = static_cast<long long>(ctx.num_sms) * 8;
      if (blocks > cap) blocks = cap;
      cfg.gridDim = dim3(static_cast<unsigned>(blocks));
      cfg.blockDim = dim3(256);
      cfg.dynamicSmemBytes = 0;
      return cudaLaunchKernelEx(&cfg, bwd_dq_convert_kernel<BF16>, reinterpret_cast<const float4*>(dQacc),
                                static_cast<uint2*>(dQ), n4, scale);
    }
  }
  {
    const long long items = static_cast<long long>(BH) * nkb;
    const int grid = static_cast<int>(items < ctx.num_sms ? items : ctx.num_sms);
    cudaError_t e;
    if (D == 64 && sp.pair) {
      e = launch_bwd_dkdv64_pair(Q, K, V, dO, LSE, delta, dK, dV, BH, M, N, scale, CAUSAL, dtype, ctx);
      if (e != cudaSuccess) return e;
    } else if constexpr (D == 64) {  // tensor memory holds the overlapped layout
      auto kern = bwd_dkdv64_kernel<BF16, CAUSAL>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, OvCfg<64>::kSmem);
      if (e != cudaSuccess) return e;
      e = launch_dependent(kern, grid, kThreadsO, OvCfg<64>::kSmem, ctx.stream, mq, mk, mv, mdo, LSE, delta,
                           static_cast<uint16_t*>(dK), static_cast<uint16_t*>(dV), BH, M, N, scale, ctx.status,
                           ctx.wait_budget_ns);
      if (e != cudaSuccess) return e;
    } else {
      auto kern = bwd_dkdv_kernel<D, BF16, CAUSAL>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (e != cudaSuccess) return e;
      e = launch_dependent(kern, grid, kThreadsB, C::kSmem, ctx.stream, mq, mk, mv, mdo, LSE, delta,
                           static_cast<uint16_t*>(dK), static_cast<uint16_t*>(dV), BH, M, N, scale, ctx.status,
                           ctx.wait_budget_ns);
      if (e != cudaSuccess) return e;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (D == 64 && sp.pair) return launch_bwd_dq64_pair(Q, K, V, dO, LSE, delta, dQ, BH, M, N, scale, CAUSAL, dtype, ctx);
  {
    auto kern = bwd_dq_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, OvCfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(BH) * nqb;
    const int grid = static_cast<int>(items < ctx.num_sms ? items : ctx.num_sms);
    e = launch_dependent(kern, grid, kThreadsO, OvCfg<D>::kSmem, ctx.stream, mq, mk, mv, mdo, LSE, delta,
                         static_cast<uint16_t*>(dQ), BH, M, N, scale, ctx.status, ctx.wait_budget_ns);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
}

}  // namespace

size_t bwd_fused_split_bytes(int num_sms) {
  return static_cast<size_t>(num_sms) * (2 * kFusedSlotFloats * sizeof(float) + kCwF * sizeof(uint32_t));
}

cudaError_t launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, float* delta, float* dQacc, int BH, int M, int N, int D,
                       float scale, bool causal, int dtype, const BwdSplit& sp, const LaunchCtx& ctx) {
  const bool bf = dtype == kBF16;
#define FA_B(DD, BB, CC)                                                                                       \
  if (D == DD && bf == BB && causal == CC)                                                                     \
    return launch_bwd_t<DD, BB, CC>(Q, K, V, O, dO, LSE, dQ, dK, dV, delta, dQacc, BH, M, N, scale, dtype, sp, ctx);
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
