// dK / dV of the backward with D = 64 on CTA pairs (tcgen05 cta_group::2).
//
// The method is the one of bwd.cu's dK/dV kernel ("06: Fused attention", attn_bwd_dkdv: P is
// recomputed from the stored log-sum-exp, dS = P o (dP - delta), dV = P^T dO, dK = scale dS^T Q).
// The layout of the work is the one the "Flash Attention" notes give for the Blackwell backward
// ("FlashAttention 4": a tile split across a CTA pair with cta_group::2, which halves the operand-B
// shared-memory traffic): a cluster of two CTAs owns 256 keys of one head, 128 in each CTA, and
// walks the query blocks of 128 once for both. Rank 0 issues every MMA for the pair with M = 256
// (one instruction covers both CTAs' key rows; each CTA's tensor memory receives its own rows):
//   S^T  = K Q^T     A: each CTA's K tile;  B: Q's 128 rows split, rows 0-63 in rank 0, 64-127 in rank 1
//   dP^T = V dO^T    the same with V and dO
//   dV  += P^T dO    A: P^T in each CTA's tensor memory;  B: dO's 64 columns split, 0-31 in rank 0,
//                    32-63 in rank 1 (MN-major, each half in the first 64 bytes of 128-byte rows)
//   dK  += dS^T Q    the same with dS^T and Q's column halves
// So each CTA streams a quarter of Q and of dO per product side (half the rows, half the columns)
// and its tensor core reads half the B operand it reads in the single-CTA kernel; the pair issues
// half the MMA instructions. The compute warps of both CTAs do exactly the single-CTA kernel's
// work on their own key rows and signal rank 0's issuers across the pair; the MMAs' completions are
// committed to the same barrier in both CTAs.
//
// Roles (352 threads): compute warps 0-7 (two per tensor-memory lane quarter, 64 query columns
// each), producer warp 8 (TMA for this CTA's halves, -LSE and -delta staging), warp 9 (allocates
// the pair's tensor memory; in rank 0 it issues S^T and dP^T), warp 10 (rank 0: issues dV and dK;
// rank 1: relays "my loads landed" to rank 0, whose MMAs read rank 1's shared memory).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bwd_common.cuh"
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kPThreads = 352;
constexpr int kPWarpProd = 8, kPWarpMma = 9, kPWarpGrad = 10;
constexpr int kPStages = 3;
constexpr int kPRowHalf = 64 * 128;  // 64 rows x 128 bytes: a row half (K-major B of S^T / dP^T)
constexpr int kPStage = 2 * kPRowHalf + 2 * kChunkB;  // Q, dO row halves; Q, dO column halves
constexpr uint32_t kPStageTx = static_cast<uint32_t>(kPStage);

struct PairHdr {
  unsigned long long fixed_full, fixed_empty;
  unsigned long long full[kPStages], empty[kPStages];
  unsigned long long peer_fixed, peer_full[kPStages];  // rank 0: rank 1's loads have landed
  unsigned long long s_full, dp_full, free1, free2, acc_full;  // MMA -> compute, committed to both CTAs
  unsigned long long sig1, sig2;  // rank 0: compute warps of both CTAs -> MMA (16 arrivals)
  unsigned long long s_read;      // rank 0: both CTAs' S^T(i) in registers (16 arrivals)
  unsigned long long mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float nlse2[kPStages][kT];  // per streamed block: -LSE * log2(e)
  alignas(16) float ndlt[kPStages][kT];   // per streamed block: -delta
};
constexpr uint32_t kPHdrBytes = (sizeof(PairHdr) + 127u) & ~127u;
constexpr int kPSmem = 1024 + static_cast<int>(kPHdrBytes) + 2 * kChunkB + kPStages * kPStage;
static_assert(kPSmem <= 232448, "shared memory budget");

// The pair's r-th item of its persistent loop (as item_of_round, over pairs).
template <bool CAUSAL>
__device__ __forceinline__ int pair_item_of_round(int r, int items) {
  const int pairs = static_cast<int>(gridDim.x >> 1), p = static_cast<int>(blockIdx.x >> 1);
  const int c = (CAUSAL && (r & 1)) ? pairs - 1 - p : p;
  const long long w = static_cast<long long>(r) * pairs + c;
  return w < items ? static_cast<int>(w) : items;
}

// TMEM: S^T [0,128), dP^T [128,256), P^T packed [256,320), dS^T packed [320,384), dV [384,448),
// dK [448,512), in both CTAs.
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kPThreads, 1)
    bwd_dkdv64_pair_kernel(const __grid_constant__ CUtensorMap tmQr, const __grid_constant__ CUtensorMap tmdOr,
                           const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                           const __grid_constant__ CUtensorMap tmQv, const __grid_constant__ CUtensorMap tmdOv,
                           const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           int have_views, const float* __restrict__ LSE, const float* __restrict__ delta,
                           uint16_t* __restrict__ dK, uint16_t* __restrict__ dV, int BH, int M, int N, float scale,
                           DevStatus* status, unsigned long long budget_ns) {
  constexpr int D = 64;
  constexpr uint32_t cS = 0, cdP = 128, cP = 256, cdS = 320, cdV = 384, cdK = 448;
  extern __shared__ uint8_t smem_raw[];
  PairHdr* hdr = reinterpret_cast<PairHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kPHdrBytes + 1023u) & ~1023u;
  const uint32_t sK = data, sV = data + kChunkB;
  auto stage = [&](int st) { return data + 2 * kChunkB + st * kPStage; };
  auto sQr = [&](int st) { return stage(st); };
  auto sdOr = [&](int st) { return stage(st) + kPRowHalf; };
  auto sQc = [&](int st) { return stage(st) + 2 * kPRowHalf; };
  auto sdOc = [&](int st) { return stage(st) + 2 * kPRowHalf + kChunkB; };
  const uint32_t rank = ptx::cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb2 = (N + 2 * kT - 1) / (2 * kT), nqb = (M + kT - 1) / kT;
  const int items = BH * nkb2;
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;
  auto item = [&](int w) {
    BwdItem it;
    // causal: the pairs of key tiles with the most query blocks first, all heads together
    int kb2;
    if (CAUSAL) {
      kb2 = w / BH;
      it.bh = w - kb2 * BH;
    } else {
      it.bh = w / nkb2;
      kb2 = w - it.bh * nkb2;
    }
    it.r0 = kb2 * 2 * kT + static_cast<int>(rank) * kT;  // this CTA's 128 keys
    it.lo = CAUSAL ? min(2 * kb2, nqb) : 0;  // query blocks before the pair's first key see none of it
    it.hi = nqb;
    return it;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->peer_fixed), 1);
    for (int st = 0; st < kPStages; ++st) {
      ptx::mbar_init(ptx::smem_u32(&hdr->full[st]), 2);  // TMA bytes + the -LSE/-delta staging
      ptx::mbar_init(ptx::smem_u32(&hdr->empty[st]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->peer_full[st]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->free1), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->free2), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig1), 16);
    ptx::mbar_init(ptx::smem_u32(&hdr->s_read), 16);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig2), 16);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[1]), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kPWarpMma) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish_pair();
  }
  if (warp == kPWarpProd && lane == 0) {
    ptx::prefetch_tmap(&tmQr);
    ptx::prefetch_tmap(&tmdOr);
    ptx::prefetch_tmap(rank == 0 && have_views ? &tmQv : &tmQ);
    ptx::prefetch_tmap(rank == 0 && have_views ? &tmdOv : &tmdO);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised, the pair's tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDkDv};
  // launched as a programmatic dependent of the delta kernel: LSE and delta are read only after it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kPWarpProd) {
    // ------------------------------------------------------------ producer (whole warp)
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
    // this CTA's column half of Q / dO: rank 0 reads columns 0-31 through a 32-column view (the box's
    // other 32 columns are out of the view and arrive as zeros), rank 1 reads columns 32-63 (the box
    // starts at column 32; its last 32 columns are out of the tensor); either way the half sits in
    // the first 64 bytes of each 128-byte row
    const CUtensorMap* mQc = rank == 0 ? (have_views ? &tmQv : &tmQ) : &tmQ;
    const CUtensorMap* mdOc = rank == 0 ? (have_views ? &tmdOv : &tmdO) : &tmdO;
    const int xc = rank == 0 ? 0 : 32;
    uint32_t it_s = 0, n_fixed = 0;  // n_fixed: K/V loads issued (lane 0)
    int n_item = 0;
    bool ok = true;
    int r = 0;
    int w = pair_item_of_round<CAUSAL>(0, items);
    BwdItem itm{};
    if (w < items) {
      itm = item(w);
      if (itm.lo < itm.hi) fetch(itm, itm.lo);
    }
    for (; w < items && ok; w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
      itm = item(w);
      if (lane == 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10);
        if (ok) {
          const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
          ptx::mbar_arrive_expect_tx(ff, 2 * kChunkB);
          ptx::tma_load_3d(sK, &tmK, ff, 0, itm.r0, itm.bh);
          ptx::tma_load_3d(sV, &tmV, ff, 0, itm.r0, itm.bh);
          ++n_fixed;
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      for (int i = itm.lo; i < itm.hi && ok; ++i, ++it_s) {
        const int st = it_s % kPStages;
        if (lane == 0)
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / kPStages) & 1u) ^ 1u, wc, 11);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(fb, kPStageTx);
          const int yr = i * kT + static_cast<int>(rank) * (kT / 2);
          ptx::tma_load_3d(sQr(st), &tmQr, fb, 0, yr, itm.bh);
          ptx::tma_load_3d(sdOr(st), &tmdOr, fb, 0, yr, itm.bh);
          ptx::tma_load_3d(sQc(st), mQc, fb, xc, i * kT, itm.bh);
          ptx::tma_load_3d(sdOc(st), mdOc, fb, xc, i * kT, itm.bh);
        }
#pragma unroll
        for (int k = 0; k < kQL; ++k) {
          hdr->nlse2[st][lane + 32 * k] = nl_v[k];
          hdr->ndlt[st][lane + 32 * k] = nd_v[k];
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fb);
        if (i + 1 < itm.hi) {
          fetch(itm, i + 1);
        } else {
          for (int r2 = r + 1, w2 = pair_item_of_round<CAUSAL>(r2, items); w2 < items;
               w2 = pair_item_of_round<CAUSAL>(++r2, items)) {
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
      for (uint32_t k = it_s > (uint32_t)kPStages ? it_s - kPStages : 0u; k < it_s; ++k)
        ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % kPStages]), (k / kPStages) & 1u, 100000000ull);
      if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
    }
  } else if ((warp == kPWarpMma || warp == kPWarpGrad) && rank == 0) {
    // ------------------------------------------------------------ MMA issuers of the pair (lane 0)
    if (lane == 0) {
      const bool scores = warp == kPWarpMma;
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(2 * kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(2 * kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, n1 = 0, n2 = 0;
      int n_item = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit_pair(ptx::smem_u32(bar)); };
      // a stage is ready once this CTA's loads and staging and rank 1's loads (relayed) are in
      auto stage_ready = [&](uint32_t k) {
        const uint32_t ph = (k / kPStages) & 1u;
        return wait(&hdr->full[k % kPStages], ph, 21) && wait(&hdr->peer_full[k % kPStages], ph, 24);
      };
      auto qk = [&](uint32_t k) {  // S^T = K Q^T over the pair's 256 keys
        const int st = k % kPStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss_pair(tmem + cS, kmajor_desc(sK, ks), kmajor_desc(sQr(st), ks), id_s, ks > 0);
        commit(&hdr->s_full);
      };
      auto vdo = [&](uint32_t k) {  // dP^T = V dO^T
        const int st = k % kPStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss_pair(tmem + cdP, kmajor_desc(sV, ks), kmajor_desc(sdOr(st), ks), id_dp, ks > 0);
        commit(&hdr->dp_full);
      };
      for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
           w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (scores) {
          if (!wait(&hdr->fixed_full, n_item & 1, 20) || !wait(&hdr->peer_fixed, n_item & 1, 25)) break;
          if (itm.lo < itm.hi) {
            ok = stage_ready(it_s);
            if (!ok) break;
            ptx::tc_fence_after();
            qk(it_s);
            vdo(it_s);
            if (itm.lo + 1 < itm.hi && !stage_ready(it_s + 1)) break;
          }
        }
        for (int i = itm.lo; i < itm.hi; ++i, ++it_s) {
          const int st = it_s % kPStages;
          const bool more = i + 1 < itm.hi;
          const bool acc = i > itm.lo;
          // scores issuer: S^T(i) read in both CTAs (its columns free for S^T(i+1) while the
          // compute warps form P); gradient issuer: P^T(i) stored in both CTAs
          ok = scores ? wait(&hdr->s_read, (n1++) & 1u, 27) : wait(&hdr->sig1, (n1++) & 1u, 22);
          if (!ok) break;
          ptx::tc_fence_after();
          if (scores) {
            if (more) qk(it_s + 1);
          } else {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)  // dV += P^T dO
              ptx::mma_f16_ts_pair(tmem + cdV, tmem + cP + ks * 8, mnmajor_desc(sdOc(st), ks), id_g, (acc || ks > 0));
            commit(&hdr->free1);
          }
          // dP^T(i) read and dS^T(i) stored, in both CTAs
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
              ptx::mma_f16_ts_pair(tmem + cdK, tmem + cdS + ks * 8, mnmajor_desc(sQc(st), ks), id_g, (acc || ks > 0));
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
  } else if (warp == kPWarpGrad && rank == 1) {
    // ------------------------------------------------------------ relay (lane 0): rank 1's loads landed
    if (lane == 0) {
      const uint32_t peer_fixed = ptx::peer_addr(ptx::smem_u32(&hdr->peer_fixed), 0);
      uint32_t it_s = 0;
      int n_item = 0;
      bool ok = true;
      for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
           w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_full), n_item & 1, wc, 26);
        if (!ok) break;
        ptx::mbar_arrive_remote(peer_fixed);
        for (int i = itm.lo; i < itm.hi && ok; ++i, ++it_s) {
          const int st = it_s % kPStages;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), (it_s / kPStages) & 1u, wc, 27);
          if (ok) ptx::mbar_arrive_remote(ptx::peer_addr(ptx::smem_u32(&hdr->peer_full[st]), 0));
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute warps: one key row per thread
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(half * 64);  // this warp's query columns [c0, c0 + 64)
    const uint32_t sig1 = ptx::peer_addr(ptx::smem_u32(&hdr->sig1), 0);
    const uint32_t s_read = ptx::peer_addr(ptx::smem_u32(&hdr->s_read), 0);
    const uint32_t sig2 = ptx::peer_addr(ptx::smem_u32(&hdr->sig2), 0);
    uint32_t it_s = 0, nb = 0, n_acc = 0;  // n_acc: items with a query block (acc_full phases)
    int n_item = 0;
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    auto signal = [&](uint32_t cl_bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(cl_bar);
    };
    for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
         w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
      const BwdItem itm = item(w);
      const int key = itm.r0 + quarter * 32 + lane;
      for (int i = itm.lo; i < itm.hi; ++i, ++it_s, ++nb) {
        const int st = it_s % kPStages;
        ok = wait_all(&hdr->s_full, nb & 1u, 30) && wait_all(&hdr->full[st], (it_s / kPStages) & 1u, 31);
        if (!ok) break;
        const float* nl = hdr->nlse2[st] + c0;
        const float* nd = hdr->ndlt[st] + c0;
        const int qb = i * kT + static_cast<int>(c0);
        const bool diag = CAUSAL && qb < key;
        float p[64];
        {
          uint32_t s[64];
          ptx::tmem_ld32(tmem + lane_sel + cS + c0, s);
          ptx::tmem_ld32(tmem + lane_sel + cS + c0 + 32, s + 32);
          ptx::tmem_wait_ld32(s);
          ptx::tmem_wait_ld32(s + 32);
          signal(s_read);  // S^T(i+1) may be computed while P is formed
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
        signal(sig1);
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
        signal(sig2);
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
  ptx::cluster_sync();  // neither CTA frees the pair's tensor memory while the other may still use it
  if (warp == kPWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

// ------------------------------------------------------------------------------- dQ on pairs
// The dQ kernel of the three-kernel backward ("06: Fused attention", attn_bwd_dq: a CTA owns query
// rows and walks the key blocks; S = Q K^T, dP = dO V^T, dS = P o (dP - delta), dQ = scale dS K) on
// CTA pairs: the pair owns 256 queries of one head, 128 in each CTA, and walks the key blocks of 128
// once for both.
//   S   = Q K^T    A: each CTA's Q tile;  B: K's 128 rows split, keys 0-63 in rank 0, 64-127 in rank 1
//   dP  = dO V^T   the same with dO and V
//   dQ += dS K     A: dS in each CTA's tensor memory;  B: K's 64 columns split, 0-31 in rank 0, 32-63
//                  in rank 1 (MN-major, each half in the first 64 bytes of 128-byte rows)
// A key block is streamed once per 256 queries (its row halves by one CTA each, its column halves
// by one CTA each), where the single-CTA kernel streams it once per 128.
constexpr int kQStages = 4;
constexpr int kQStage = 2 * kPRowHalf + kChunkB;  // K and V row halves, K column half
constexpr uint32_t kQStageTx = static_cast<uint32_t>(kQStage);

struct PairDqHdr {
  unsigned long long fixed_full, fixed_empty, peer_fixed;
  unsigned long long full[kQStages], empty[kQStages], peer_full[kQStages];
  unsigned long long s_full, dp_full, free2, acc_full;  // MMA -> compute, committed to both CTAs
  unsigned long long sig1, sig2;                        // rank 0: compute warps of both CTAs -> MMA
  unsigned long long mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kQHdrBytes = (sizeof(PairDqHdr) + 127u) & ~127u;
constexpr int kQSmem = 1024 + static_cast<int>(kQHdrBytes) + 2 * kChunkB + kQStages * kQStage;
static_assert(kQSmem <= 232448, "shared memory budget");

// TMEM: S [0,128), dP [128,256), dS packed [256,320), dQ [320,384), in both CTAs.
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kPThreads, 1)
    bwd_dq64_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmVr,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmKv,
                         int have_views, const float* __restrict__ LSE, const float* __restrict__ delta,
                         uint16_t* __restrict__ dQ, int BH, int M, int N, float scale, DevStatus* status,
                         unsigned long long budget_ns) {
  constexpr int D = 64;
  constexpr uint32_t cS = 0, cdP = 128, cdS = 256, cdQ = 320;
  extern __shared__ uint8_t smem_raw[];
  PairDqHdr* hdr = reinterpret_cast<PairDqHdr*>(smem_raw);
  const uint32_t data = (ptx::smem_u32(smem_raw) + kQHdrBytes + 1023u) & ~1023u;
  const uint32_t sQ = data, sdO = data + kChunkB;
  auto stage = [&](int st) { return data + 2 * kChunkB + st * kQStage; };
  auto sKr = [&](int st) { return stage(st); };
  auto sVr = [&](int st) { return stage(st) + kPRowHalf; };
  auto sKc = [&](int st) { return stage(st) + 2 * kPRowHalf; };
  const uint32_t rank = ptx::cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + kT - 1) / kT, nqb2 = (M + 2 * kT - 1) / (2 * kT);
  const int items = BH * nqb2;
  const float sl2 = fmaxf(fabsf(scale), 1e-30f) * kLog2eB;
  const uint32_t neg_a = scale < 0.f ? ptx::kNegateA : 0u;
  auto item = [&](int w) {
    BwdItem it;
    const int qb2_rev = w / BH;  // causal: the heaviest (last) pairs of query tiles first
    it.bh = w - qb2_rev * BH;
    const int qb2 = CAUSAL ? nqb2 - 1 - qb2_rev : qb2_rev;
    it.r0 = qb2 * 2 * kT + static_cast<int>(rank) * kT;  // this CTA's 128 queries
    it.lo = 0;
    it.hi = CAUSAL ? min(nkb, (qb2 * 2 * kT + 2 * kT - 1) / kT + 1) : nkb;  // up to the pair's last query
    return it;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->fixed_empty), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->peer_fixed), 1);
    for (int st = 0; st < kQStages; ++st) {
      ptx::mbar_init(ptx::smem_u32(&hdr->full[st]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->empty[st]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->peer_full[st]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->free2), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig1), 16);
    ptx::mbar_init(ptx::smem_u32(&hdr->sig2), 16);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[1]), 1);
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kPWarpMma) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish_pair();
  }
  if (warp == kPWarpProd && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmdO);
    ptx::prefetch_tmap(&tmKr);
    ptx::prefetch_tmap(&tmVr);
    ptx::prefetch_tmap(rank == 0 && have_views ? &tmKv : &tmK);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised, the pair's tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernBwdDq};
  // launched as a programmatic dependent of the dK/dV kernel: global memory only after it completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kPWarpProd) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      const CUtensorMap* mKc = rank == 0 ? (have_views ? &tmKv : &tmK) : &tmK;
      const int xc = rank == 0 ? 0 : 32;
      uint32_t it_s = 0, n_fixed = 0;  // n_fixed: Q/dO loads issued
      int n_item = 0;
      bool ok = true;
      for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
           w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_empty), (n_item & 1) ^ 1, wc, 10)) break;
        const uint32_t ff = ptx::smem_u32(&hdr->fixed_full);
        ptx::mbar_arrive_expect_tx(ff, 2 * kChunkB);
        ptx::tma_load_3d(sQ, &tmQ, ff, 0, itm.r0, itm.bh);
        ptx::tma_load_3d(sdO, &tmdO, ff, 0, itm.r0, itm.bh);
        ++n_fixed;
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % kQStages;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->empty[st]), ((it_s / kQStages) & 1u) ^ 1u, wc, 11);
          if (!ok) break;
          const uint32_t fb = ptx::smem_u32(&hdr->full[st]);
          ptx::mbar_arrive_expect_tx(fb, kQStageTx);
          const int yr = j * kT + static_cast<int>(rank) * (kT / 2);
          ptx::tma_load_3d(sKr(st), &tmKr, fb, 0, yr, itm.bh);
          ptx::tma_load_3d(sVr(st), &tmVr, fb, 0, yr, itm.bh);
          ptx::tma_load_3d(sKc(st), mKc, fb, xc, j * kT, itm.bh);
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = it_s > (uint32_t)kQStages ? it_s - kQStages : 0u; k < it_s; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->full[k % kQStages]), (k / kQStages) & 1u, 100000000ull);
        if (n_fixed > 0u) ptx::mbar_wait_drain(ptx::smem_u32(&hdr->fixed_full), (n_fixed - 1u) & 1u, 100000000ull);
      }
    }
  } else if ((warp == kPWarpMma || warp == kPWarpGrad) && rank == 0) {
    // ------------------------------------------------------------ MMA issuers of the pair (lane 0)
    if (lane == 0) {
      const bool scores = warp == kPWarpMma;
      constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
      const uint32_t id_dp = ptx::idesc_f32acc(2 * kT, kT, fmt, fmt, false, false);  // dP: never negated
      const uint32_t id_s = id_dp | neg_a;
      constexpr uint32_t id_g = ptx::idesc_f32acc(2 * kT, D, fmt, fmt, false, true);
      uint32_t it_s = 0, n1 = 0, n2 = 0;
      int n_item = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit_pair(ptx::smem_u32(bar)); };
      auto stage_ready = [&](uint32_t k) {
        const uint32_t ph = (k / kQStages) & 1u;
        return wait(&hdr->full[k % kQStages], ph, 21) && wait(&hdr->peer_full[k % kQStages], ph, 24);
      };
      auto qk = [&](uint32_t k) {  // S = Q K^T over the pair's 256 queries
        const int st = k % kQStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss_pair(tmem + cS, kmajor_desc(sQ, ks), kmajor_desc(sKr(st), ks), id_s, ks > 0);
        commit(&hdr->s_full);
      };
      auto dov = [&](uint32_t k) {  // dP = dO V^T
        const int st = k % kQStages;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_f16_ss_pair(tmem + cdP, kmajor_desc(sdO, ks), kmajor_desc(sVr(st), ks), id_dp, ks > 0);
        commit(&hdr->dp_full);
      };
      for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
           w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        if (scores) {
          if (!wait(&hdr->fixed_full, n_item & 1, 20) || !wait(&hdr->peer_fixed, n_item & 1, 25)) break;
          if (itm.lo < itm.hi) {
            ok = stage_ready(it_s);
            if (!ok) break;
            ptx::tc_fence_after();
            qk(it_s);
            dov(it_s);
            if (itm.lo + 1 < itm.hi && !stage_ready(it_s + 1)) break;
          }
        }
        for (int j = itm.lo; j < itm.hi; ++j, ++it_s) {
          const int st = it_s % kQStages;
          const bool more = j + 1 < itm.hi;
          if (scores) {
            // S(j) read in both CTAs
            ok = wait(&hdr->sig1, (n1++) & 1u, 22);
            if (!ok) break;
            ptx::tc_fence_after();
            if (more) qk(it_s + 1);
          }
          // dP(j) read and dS(j) stored in both CTAs
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
              ptx::mma_f16_ts_pair(tmem + cdQ, tmem + cdS + ks * 8, mnmajor_desc(sKc(st), ks), id_g,
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
  } else if (warp == kPWarpGrad && rank == 1) {
    // ------------------------------------------------------------ relay (lane 0): rank 1's loads landed
    if (lane == 0) {
      const uint32_t peer_fixed = ptx::peer_addr(ptx::smem_u32(&hdr->peer_fixed), 0);
      uint32_t it_s = 0;
      int n_item = 0;
      bool ok = true;
      for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
           w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
        const BwdItem itm = item(w);
        ok = ptx::mbar_wait(ptx::smem_u32(&hdr->fixed_full), n_item & 1, wc, 26);
        if (!ok) break;
        ptx::mbar_arrive_remote(peer_fixed);
        for (int j = itm.lo; j < itm.hi && ok; ++j, ++it_s) {
          const int st = it_s % kQStages;
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->full[st]), (it_s / kQStages) & 1u, wc, 27);
          if (ok) ptx::mbar_arrive_remote(ptx::peer_addr(ptx::smem_u32(&hdr->peer_full[st]), 0));
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute warps: one query row per thread
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t c0 = static_cast<uint32_t>(half * 64);  // this warp's key columns [c0, c0 + 64)
    const uint32_t sig1 = ptx::peer_addr(ptx::smem_u32(&hdr->sig1), 0);
    const uint32_t sig2 = ptx::peer_addr(ptx::smem_u32(&hdr->sig2), 0);
    uint32_t nb = 0;
    int n_item = 0;
    bool ok = true;
    auto wait_all = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
      const bool r = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site));
      ptx::tc_fence_after();
      return r;
    };
    auto signal = [&](uint32_t cl_bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(cl_bar);
    };
    for (int r = 0, w = pair_item_of_round<CAUSAL>(0, items); w < items && ok;
         w = pair_item_of_round<CAUSAL>(++r, items), ++n_item) {
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
        signal(sig1);  // S(j) read: the next S may be computed
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
        signal(sig2);
      }
      if (!ok) break;
      ok = wait_all(&hdr->acc_full, n_item & 1, 33);
      if (!ok) break;
      const bool none = itm.lo >= itm.hi;
      uint32_t a[32];
      ptx::tmem_ld32(tmem + lane_sel + cdQ + 32 * half, a);
      ptx::tmem_wait_ld32(a);
      uint32_t h[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        h[k] = none ? 0u : pack2<BF16>(__uint_as_float(a[2 * k]) * scale, __uint_as_float(a[2 * k + 1]) * scale);
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dQ + g * D + 32 * half);
#pragma unroll
        for (int v = 0; v < 4; ++v) d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
      }
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // neither CTA frees the pair's tensor memory while the other may still use it
  if (warp == kPWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

template <bool BF16, bool CAUSAL>
cudaError_t launch_dq_pair_t(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                             const float* delta, void* dQ, int BH, int M, int N, float scale, int dtype,
                             const LaunchCtx& ctx) {
  constexpr int D = 64;
  CUtensorMap mq, mdo, mkr, mvr, mk, mkv;
  if (!make_tmap_3d(&mq, Q, dtype, D, M, BH, 64, kT) || !make_tmap_3d(&mdo, dO, dtype, D, M, BH, 64, kT) ||
      !make_tmap_3d(&mkr, K, dtype, D, N, BH, 64, kT / 2) || !make_tmap_3d(&mvr, V, dtype, D, N, BH, 64, kT / 2) ||
      !make_tmap_3d(&mk, K, dtype, D, N, BH, 64, kT))
    return cudaErrorInvalidValue;
  const int have_views = make_tmap_3d_view(&mkv, K, dtype, 32, D, N, BH, 64, kT);
  if (!have_views) mkv = mk;
  auto kern = bwd_dq64_pair_kernel<BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kQSmem;
  cfg.stream = ctx.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * static_cast<unsigned>(ctx.num_sms / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs = n > 0 ? n : 1;
  }
  const long long items = static_cast<long long>(BH) * ((M + 2 * kT - 1) / (2 * kT));
  const int pairs = static_cast<int>(items < max_pairs ? items : max_pairs);
  cfg.gridDim = dim3(2 * static_cast<unsigned>(pairs));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mq, mdo, mkr, mvr, mk, mkv, have_views, LSE, delta,
                            static_cast<uint16_t*>(dQ), BH, M, N, scale, ctx.status, ctx.wait_budget_ns);
}

template <bool BF16, bool CAUSAL>
cudaError_t launch_pair_t(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                          const float* delta, void* dK, void* dV, int BH, int M, int N, float scale, int dtype,
                          const LaunchCtx& ctx) {
  constexpr int D = 64;
  CUtensorMap mqr, mdor, mq, mdo, mqv, mdov, mk, mv;
  if (!make_tmap_3d(&mqr, Q, dtype, D, M, BH, 64, kT / 2) || !make_tmap_3d(&mdor, dO, dtype, D, M, BH, 64, kT / 2) ||
      !make_tmap_3d(&mq, Q, dtype, D, M, BH, 64, kT) || !make_tmap_3d(&mdo, dO, dtype, D, M, BH, 64, kT) ||
      !make_tmap_3d(&mk, K, dtype, D, N, BH, 64, kT) || !make_tmap_3d(&mv, V, dtype, D, N, BH, 64, kT))
    return cudaErrorInvalidValue;
  // 32-column views of Q and dO (rows of 64 elements): rank 0's column half without reading the
  // other half; if the driver refuses them, rank 0 reads whole rows instead (same result)
  const int have_views = make_tmap_3d_view(&mqv, Q, dtype, 32, D, M, BH, 64, kT) &&
                         make_tmap_3d_view(&mdov, dO, dtype, 32, D, M, BH, 64, kT);
  if (!have_views) {
    mqv = mq;
    mdov = mdo;
  }
  auto kern = bwd_dkdv64_pair_kernel<BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = ctx.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // pairs that fit at once (one CTA per SM): a persistent grid of that many clusters
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * static_cast<unsigned>(ctx.num_sms / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs = n > 0 ? n : 1;
  }
  const long long items = static_cast<long long>(BH) * ((N + 2 * kT - 1) / (2 * kT));
  const int pairs = static_cast<int>(items < max_pairs ? items : max_pairs);
  cfg.gridDim = dim3(2 * static_cast<unsigned>(pairs));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mqr, mdor, mq, mdo, mqv, mdov, mk, mv, have_views, LSE, delta,
                            static_cast<uint16_t*>(dK), static_cast<uint16_t*>(dV), BH, M, N, scale, ctx.status,
                            ctx.wait_budget_ns);
}

}  // namespace

cudaError_t launch_bwd_dkdv64_pair(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                                   const float* delta, void* dK, void* dV, int BH, int M, int N, float scale,
                                   bool causal, int dtype, const LaunchCtx& ctx) {
  const bool bf = dtype == kBF16;
  if (!bf && !causal) return launch_pair_t<false, false>(Q, K, V, dO, LSE, delta, dK, dV, BH, M, N, scale, dtype, ctx);
  if (!bf && causal) return launch_pair_t<false, true>(Q, K, V, dO, LSE, delta, dK, dV, BH, M, N, scale, dtype, ctx);
  if (bf && !causal) return launch_pair_t<true, false>(Q, K, V, dO, LSE, delta, dK, dV, BH, M, N, scale, dtype, ctx);
  return launch_pair_t<true, true>(Q, K, V, dO, LSE, delta, dK, dV, BH, M, N, scale, dtype, ctx);
}

cudaError_t launch_bwd_dq64_pair(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                                 const float* delta, void* dQ, int BH, int M, int N, float scale, bool causal,
                                 int dtype, const LaunchCtx& ctx) {
  const bool bf = dtype == kBF16;
  if (!bf && !causal) return launch_dq_pair_t<false, false>(Q, K, V, dO, LSE, delta, dQ, BH, M, N, scale, dtype, ctx);
  if (!bf && causal) return launch_dq_pair_t<false, true>(Q, K, V, dO, LSE, delta, dQ, BH, M, N, scale, dtype, ctx);
  if (bf && !causal) return launch_dq_pair_t<true, false>(Q, K, V, dO, LSE, delta, dQ, BH, M, N, scale, dtype, ctx);
  return launch_dq_pair_t<true, true>(Q, K, V, dO, LSE, delta, dQ, BH, M, N, scale, dtype, ctx);
}

}  // namespace fa
