// Forward prefill for fp16 / bf16 inputs with head dimension 64.
//
// Same method as the general half-precision forward (FlashAttention-2's
// forward: running max m, denominator l and unnormalised O carried across key
// blocks, one division at the end, L = m + log l; the FA4 conditional
// rescale), with a tensor-memory plan that only fits when D = 64:
//
//   S0 [0,128)  S1 [128,256)  P0 [256,320)  P1 [320,384)  O0 [384,448)  O1 [448,512)
//
// P has columns of its own, so a tile's scores are released as soon as the
// softmax threads hold them in registers (a row of 128 f32 scores per thread):
// S_t(j+2) = Q_t K_{j+2}^T is computed while the softmax of block j+1 runs, and
// O_t += P_t(j) V_j as soon as P_t(j) is stored. A tile's softmax therefore
// never waits for its own MMAs.
//
// Each tile has its own MMA-issuing thread (warps 9 and 10). A tcgen05.mma issue
// blocks until the tensor pipe takes it, so an issuer's waits and commits leave
// the pipe idle unless the other tile's issuer has MMAs queued: two issuers
// overlap that bookkeeping. P of a block is formed and handed over in two
// halves of 64 keys: P V over the first half runs while the softmax forms the
// second, and P V over the second half while the softmax reads the next scores
// and forms its first half, so a tile's softmax never waits for P V either.
// Per tile the issue order is S(0), S(1), then per block j: P_a V(j), P_b V(j),
// S(j+2). The softmax signals two barriers per block (sm_a: first half of P(j)
// stored; sm_b: second half of P(j-1) stored and S(j) read); K and V of a block
// land on one barrier.
//
// Per block and row: the block maximum first (from registers), a warp-uniform
// decision whether any row's maximum moved by more than 2^8 (then O, l are
// rescaled in place), then P = 2^(s*c - m) packed to halves. O is divided by
// the sum of the half-rounded weights that multiplied V (so it is a convex
// combination of V rows); LSE uses the exact f32 sum.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "fwd_common.cuh"
#include "fwd_split.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using fwdc::fadd2;
using fwdc::ffma2;
using fwdc::fmax3;
using fwdc::kBM;
using fwdc::kBN;
using fwdc::mask32;
using fwds::kPairRows;
using fwds::kSlotFloats;
using fwds::Piece;
using fwds::Schedule;
using fwds::split_bounds;
using fwds::SplitBounds;
using fwds::units_before;

constexpr int kD = 64;
constexpr int kTile = kBM * kD * 2;  // 16 KB: one 128-row x 64-column half tile (128-byte rows)
constexpr int kStages = 4;           // K/V ring depth (blocks j..j+2 in use, j+3 loading)
constexpr int kQBuf = 2;             // Q pair buffers
// softmax 0-3 (tile 0), 4-7 (tile 1), producer 8, MMA issuers 9 (tile 0) and 10 (tile 1),
// epilogue helper 11. Three warps share an SM sub-partition (16K registers): 168 registers a thread.
constexpr int kThreads = 384;
constexpr int kWarpProd = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpEpi = 11;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSmemData = kQBuf * 2 * kTile + kStages * 2 * kTile;
constexpr int kSmemBytes = 1024 + 1024 + kSmemData;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// tensor-memory columns
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;

struct Hdr {
  unsigned long long q_full[kQBuf], q_empty[kQBuf];  // q_empty: the helper is done with the buffer
  // epi[qb][t]: tile t's 4 softmax warps are done with a piece held in Q buffer qb (O rows written
  // into the buffer, or the partial written to global memory). One barrier per buffer, so the
  // next arrival on it needs q_empty[qb] first and the helper is never two phases behind.
  unsigned long long epi[kQBuf][2];
  unsigned long long kv_full[kStages], kv_empty[kStages];  // kv_empty: one commit per issuer
  unsigned long long s_full[2];   // S_t(j) computed
  unsigned long long sm_a[2];     // softmax of tile t: first half of P_t(j) stored (4 warps)
  unsigned long long sm_b[2];     // softmax of tile t: second half of P_t(j-1) stored, S_t(j) read (4 warps)
  unsigned long long p_free_a[2]; // P V over the first half of block j computed
  unsigned long long p_free_b[2]; // P V over the second half of block j computed (O_t holds block j)
  unsigned long long o_full[2];   // the pair's last P_t V computed
  unsigned long long mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_d64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, float* __restrict__ LSE, int BH,
                   int M, int N, float scale_log2_signed, float* __restrict__ ws, uint32_t* __restrict__ flags, uint32_t epoch,
                   DevStatus* status, unsigned long long budget_ns, int inject,
                   const __grid_constant__ SplitBounds bounds) {
  extern __shared__ uint8_t smem_raw[];
  Hdr* hdr = reinterpret_cast<Hdr*>(smem_raw);
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t data_u32 = (raw_u32 + 1024u + 1023u) & ~1023u;  // 1024-aligned for the swizzle atoms
  auto q_addr = [&](int qb, int t) { return data_u32 + (qb * 2 + t) * kTile; };
  auto k_addr = [&](int st) { return data_u32 + kQBuf * 2 * kTile + st * 2 * kTile; };
  auto v_addr = [&](int st) { return k_addr(st) + kTile; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_pairs = (M + 2 * kBM - 1) / (2 * kBM);
  const int nkb = (N + kBN - 1) / kBN;
  const bool split = ws != nullptr;
  const uint32_t* bnd = split && bounds.s[gridDim.x] != 0u ? bounds.s : nullptr;
  // scale < 0: the score product is negated in the tensor core and the softmax scales by |scale|.
  // |scale| is kept above 1e-30 so that a masked score (-inf) times it stays -inf when scale = 0
  // (every visible weight is then exp2 of about 0, i.e. 1).
  const bool neg_scale = scale_log2_signed < 0.f;
  const float scale_log2 = fmaxf(fabsf(scale_log2_signed), 1e-30f);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQBuf; ++i) {
      ptx::mbar_init(ptx::smem_u32(&hdr->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->q_empty[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->epi[i][0]), 4);
      ptx::mbar_init(ptx::smem_u32(&hdr->epi[i][1]), 4);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&hdr->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->sm_a[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&hdr->sm_b[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&hdr->p_free_a[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->p_free_b[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->o_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->mma_done[i]), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_empty[i]), 2);
    }
    hdr->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(&hdr->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    // where the start weighs most (whole pairs, or split shares of at most 128 units), the first
    // piece's Q tiles and first key blocks start towards L2 while the CTA sets up: a dependent
    // launch's set-up runs on the SMs the previous kernel has left, during that kernel's tail.
    // (A prefetch only warms L2, where the previous kernel's writes land too.) At B4 H12 N2048
    // (40 units a CTA) 63.2 -> 62.0 us back to back.
    Schedule<CAUSAL> first(split, BH, num_pairs, nkb, bnd);
    Piece p0;
    if ((!split || first.e - first.u <= 128u) && first.next(p0, split, BH, num_pairs, nkb)) {
      for (int t = 0; t < 2; ++t) ptx::tma_prefetch_l2_3d(&tmQ, 0, p0.q0 + t * kBM, p0.bh);
      const int nb = p0.nb1 < kStages ? p0.nb1 : kStages;
      for (int j = 0; j < nb; ++j) {
        ptx::tma_prefetch_l2_3d(&tmK, 0, (p0.jb + j) * kBN, p0.bh);
        ptx::tma_prefetch_l2_3d(&tmV, 0, (p0.jb + j) * kBN, p0.bh);
      }
    }
  }
  if (warp == kWarpEpi && lane == 0) ptx::prefetch_tmap(&tmO);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernFwd};
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_it = 0;
      const bool skip_first = inject == kInjectFwdStage && blockIdx.x == 0;
      int it = 0;
      bool ok = true;
      Schedule<CAUSAL> sch(split, BH, num_pairs, nkb, bnd);
      Piece ti;
      for (; ok && sch.next(ti, split, BH, num_pairs, nkb); ++it) {
        const int qb = it % kQBuf;
        const uint32_t qph = static_cast<uint32_t>(it / kQBuf) & 1u;
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->q_empty[qb]), qph ^ 1u, wc, 10)) break;
        const uint32_t qf = ptx::smem_u32(&hdr->q_full[qb]);
        ptx::mbar_arrive_expect_tx(qf, 2 * kTile);
        for (int t = 0; t < 2; ++t) ptx::tma_load_3d(q_addr(qb, t), &tmQ, qf, 0, ti.q0 + t * kBM, ti.bh);
        for (int j = 0; j < ti.nb1; ++j, ++kv_it) {
          const int st = kv_it % kStages;
          const uint32_t ph = (kv_it / kStages) & 1u;
          if (!ptx::mbar_wait(ptx::smem_u32(&hdr->kv_empty[st]), ph ^ 1u, wc, 11)) {
            ok = false;
            break;
          }
          // test-only fault injection: the first CTA never fills the first stage of K/V, so the
          // waits on it run out and the launch reports a timeout (no fault, no trap)
          if (kv_it == 0 && skip_first) continue;
          const uint32_t f = ptx::smem_u32(&hdr->kv_full[st]);
          ptx::mbar_arrive_expect_tx(f, 2 * kTile);
          ptx::tma_load_3d(k_addr(st), &tmK, f, 0, (ti.jb + j) * kBN, ti.bh);
          ptx::tma_load_3d(v_addr(st), &tmV, f, 0, (ti.jb + j) * kBN, ti.bh);
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = kv_it > (uint32_t)kStages ? kv_it - kStages : 0u; k < kv_it; ++k) {
          if (!(k == 0 && skip_first))
            ptx::mbar_wait_drain(ptx::smem_u32(&hdr->kv_full[k % kStages]), (k / kStages) & 1u, 100000000ull);
        }
        // Q loads issued: one per piece taken (it)
        for (int k = it > kQBuf ? it - kQBuf : 0; k < it; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->q_full[k % kQBuf]), static_cast<uint32_t>(k / kQBuf) & 1u, 100000000ull);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpMma + 1) {
    // ------------------------------------------------------------ MMA issuer of tile t (lane 0)
    constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
    const uint32_t idesc_qk = ptx::idesc_f32acc(kBM, kBN, fmt, fmt, false, false) | (neg_scale ? ptx::kNegateA : 0u);
    constexpr uint32_t idesc_pv = ptx::idesc_f32acc(kBM, kD, fmt, fmt, false, true);
    const int t = warp - kWarpMma;
    if (lane == 0) {
      uint32_t kv_base = 0;  // ring index of the pair's first key block
      uint32_t n_a = 0, n_b = 0;  // softmax arrivals consumed on sm_a / sm_b (all pairs)
      int it = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      const uint32_t dS = tmem + kColS + t * kBN;
      const uint32_t dO = tmem + kColO + t * kD;
      const uint32_t aP = tmem + kColP + t * (kBN / 2);
      Schedule<CAUSAL> sch(split, BH, num_pairs, nkb, bnd);
      Piece ti;
      for (; ok && sch.next(ti, split, BH, num_pairs, nkb); ++it) {
        const int qb = it % kQBuf;
        const int nb = t == 0 ? ti.nb0 : ti.nb1;
        if (!wait(&hdr->q_full[qb], static_cast<uint32_t>(it / kQBuf) & 1u, 20)) break;
        auto kv_ready = [&](int j) {
          const uint32_t kv = kv_base + j;
          return wait(&hdr->kv_full[kv % kStages], (kv / kStages) & 1u, 21);
        };
        auto arrival_a = [&]() { return wait(&hdr->sm_a[t], (n_a++) & 1u, 22); };
        auto arrival_b = [&]() { return wait(&hdr->sm_b[t], (n_b++) & 1u, 23); };
        // S_t(j) = Q_t K_j^T
        auto qk = [&](int j) {
          ptx::tc_fence_after();
          const uint64_t a0 = ptx::sdesc_sw128(q_addr(qb, t), 16, 1024);
          const uint64_t b0 = ptx::sdesc_sw128(k_addr((kv_base + j) % kStages), 16, 1024);
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) ptx::mma_f16_ss(dS, a0 + 2 * ks, b0 + 2 * ks, idesc_qk, ks > 0 ? 1u : 0u);
          commit(&hdr->s_full[t]);
        };
        // O_t (+)= P_t(j) V_j over keys [64h, 64h + 64) of the block
        auto pv = [&](int j, int h) {
          ptx::tc_fence_after();
          const uint64_t b0 = ptx::sdesc_sw128(v_addr((kv_base + j) % kStages), kTile, 1024);
#pragma unroll
          for (int ks = 4 * h; ks < 4 * h + 4; ++ks)
            ptx::mma_f16_ts(dO, aP + ks * 8, b0 + static_cast<uint64_t>((ks * 2048) >> 4), idesc_pv,
                            (j > 0 || ks > 0) ? 1u : 0u);
          commit(h == 0 ? &hdr->p_free_a[t] : &hdr->p_free_b[t]);
          if (h == 1 && j == nb - 1) commit(&hdr->o_full[t]);
        };
        ok = kv_ready(0);
        if (ok) qk(0);
        // S_t(0) read (only signalled when there is an S_t(1) to compute: with one block the
        // next arrival would not depend on this thread, and a waiter two phases behind a
        // barrier never sees its phase complete)
        if (ok && nb > 1) {
          ok = arrival_b() && kv_ready(1);
          if (ok) qk(1);
        }
        for (int j = 0; j < nb && ok; ++j) {
          // K_{j+2} is normally long loaded: its barrier is checked while the softmax forms
          // P_t(j), not between the softmax's signal and the MMAs it releases
          if (j + 2 < nb) {
            ok = kv_ready(j + 2);
            if (!ok) break;
          }
          ok = arrival_a();  // first half of P_t(j) stored
          if (!ok) break;
          pv(j, 0);
          ok = arrival_b();  // second half of P_t(j) stored (and S_t(j+1) read)
          if (!ok) break;
          pv(j, 1);
          if (j + 2 < nb) qk(j + 2);
          commit(&hdr->kv_empty[(kv_base + j) % kStages]);  // this tile is done with K_j, V_j
        }
        // blocks of the pair this tile does not use (causal): release them once loaded
        for (int j = nb; j < ti.nb1 && ok; ++j) {
          ok = kv_ready(j);
          if (ok) commit(&hdr->kv_empty[(kv_base + j) % kStages]);
        }
        kv_base += ti.nb1;
      }
      // every MMA issued by this thread has completed once mma_done flips
      commit(&hdr->mma_done[t]);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[t]), 0u, 1000000000ull);
    }
  } else if (warp == kWarpEpi) {
    // ------------------------------------------------------------ epilogue helper (lane 0)
    // Per piece, once a tile's softmax warps are done with it: the TMA store of the tile's O from
    // its Q buffer, or (a partial) the fence and the ready flags that publish the partial the
    // warps wrote; then, both tiles done, the Q buffer's release. None of this waits on the
    // softmax warps' critical path.
    if (lane == 0) {
      Schedule<CAUSAL> sch(split, BH, num_pairs, nkb, bnd);
      Piece ti;
      for (int it = 0; sch.next(ti, split, BH, num_pairs, nkb); ++it) {
        const int qb = it % kQBuf;
        const uint32_t ph = static_cast<uint32_t>(it / kQBuf) & 1u;
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t) {
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->epi[qb][t]), ph, wc, 37);
          if (ok && ti.kind != 2) {
            ptx::tma_store_3d(&tmO, q_addr(qb, t), 0, ti.q0 + t * kBM, ti.bh);
            ptx::bulk_commit();
          }
        }
        if (!ok) break;
        if (ti.kind == 2) {
          // the softmax warps' partial writes were ordered before their epi arrivals, which this
          // thread has observed: a gpu-scope fence from here, then the flag stores, publishes them
          // (cumulativity). One fence serves all eight flags: a release store each would fence
          // again, eight round trips in a row (several us per partial on small shares).
          __threadfence();
          // (test-only fault injection: CTA 1 never publishes, so the CTA merging its partial
          // gives up its bounded wait on the flags and the launch reports a timeout)
          if (!(inject == kInjectFwdFlag && blockIdx.x == 1))
            for (int w = 0; w < 8; ++w) ptx::st_relaxed_u32(flags + static_cast<size_t>(blockIdx.x) * 8 + w, epoch);
        } else {
          ptx::bulk_wait_read();  // both stores have read the buffer
        }
        ptx::mbar_arrive(ptx::smem_u32(&hdr->q_empty[qb]));
      }
      ptx::bulk_wait_all();  // the O stores have completed
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (one row per thread)
    const int t = warp >> 2;  // tile of the pair
    const int wq = warp & 3;  // TMEM lane quarter
    const uint32_t lane_sel = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_sel + kColS + t * kBN;
    const uint32_t tP = tmem + lane_sel + kColP + t * (kBN / 2);
    const uint32_t tO = tmem + lane_sel + kColO + t * kD;
    const uint32_t s_full = ptx::smem_u32(&hdr->s_full[t]);
    const uint32_t sm_a = ptx::smem_u32(&hdr->sm_a[t]);
    const uint32_t sm_b = ptx::smem_u32(&hdr->sm_b[t]);
    const uint32_t p_free_a = ptx::smem_u32(&hdr->p_free_a[t]);
    const uint32_t p_free_b = ptx::smem_u32(&hdr->p_free_b[t]);
    const uint32_t o_full = ptx::smem_u32(&hdr->o_full[t]);
    uint32_t nblk = 0u;  // blocks processed by this tile slot (all pairs)
    uint32_t o_ph = 0u;
    bool ok = true;
    Schedule<CAUSAL> sch(split, BH, num_pairs, nkb, bnd);
    Piece ti;
    int it = 0;          // pieces taken (Q buffer = it % kQBuf)
    for (; ok && sch.next(ti, split, BH, num_pairs, nkb); ++it) {
      const int nbt = t == 0 ? ti.nb0 : ti.nb1;
      const int qb = it % kQBuf;
      const int row = ti.q0 + t * kBM + wq * 32 + lane;  // query index within the head
      float m2 = -INFINITY;  // running max of scale*log2(e)*s (stale by at most 2^8)
      float l = 0.f;         // sum of the half-rounded weights (normalises O)
      float le = 0.f;        // sum of the exact f32 weights (gives LSE)
      for (int j = 0; j < nbt; ++j, ++nblk) {
        // warp-uniform outcome: the tcgen05 loads below are .aligned
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(s_full, nblk & 1u, wc, 30));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t r[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) ptx::tmem_ld32(tS + c, r + c);
#pragma unroll
        for (int c = 0; c < kBN; c += 32) ptx::tmem_wait_ld32(r + c);
        // the scores are in registers (the tile's S columns may be overwritten) and the
        // previous block's second half of P is stored (waited at the end of that block)
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && (j > 0 || nbt > 1)) ptx::mbar_arrive(sm_b);

        const int kbase = (ti.jb + j) * kBN;
        if ((kbase + kBN > N) || (CAUSAL && kbase + kBN - 1 > ti.q0 + t * kBM)) {
#pragma unroll
          for (int c = 0; c < kBN; c += 32) mask32<CAUSAL>(r + c, kbase + c, N, row);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < kBN; i += 8) {
          mx0 = fmax3(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
          mx1 = fmax3(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
          mx2 = fmax3(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
          mx3 = fmax3(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
        }
        const float mxs = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
        // warp-uniform: does any row's maximum move by more than the threshold?
        const bool rescale = j == 0 || __any_sync(0xFFFFFFFFu, mxs > m2 + kRescaleThreshold);
        float corr = 1.f;
        if (rescale) {
          const float m_new = fmaxf(m2, mxs);
          corr = m_new == -INFINITY ? 1.f : ptx::ex2(m2 - m_new);
          l *= corr;
          le *= corr;
          m2 = m_new;
        }
        const float neg_m = m2 == -INFINITY ? 0.f : -m2;
        const float2 c2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(neg_m, neg_m);
        float2 se = make_float2(0.f, 0.f);
        float sr0 = 0.f, sr1 = 0.f;
        // P over keys [c, c + 32): packed halves stored to columns [c/2, c/2 + 16)
        auto p_piece = [&](int c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x =
                ffma2(make_float2(__uint_as_float(r[c + 2 * i]), __uint_as_float(r[c + 2 * i + 1])), c2, nm2);
            const float a = ptx::ex2(x.x), b = ptx::ex2(x.y);
            se = fadd2(se, make_float2(a, b));
            pk[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
            if (BF16)
              ptx::add_bf16x2_to_f32(pk[i], sr0, sr1);
            else
              ptx::add_f16x2_to_f32(pk[i], sr0, sr1);
          }
          ptx::tmem_st16(tP + c / 2, pk);
        };
        // first half: P V over it from the previous block must have completed
        if (nblk > 0u) {
          ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(p_free_a, (nblk - 1u) & 1u, wc, 32));
          if (!ok) break;
          ptx::tc_fence_after();
        }
        p_piece(0);
        p_piece(32);
        bool b_done = nblk == 0u;
        if (rescale && j > 0) {  // O holds earlier blocks: rescale it once the previous P V has completed
          ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(p_free_b, (nblk - 1u) & 1u, wc, 33));
          if (!ok) break;
          ptx::tc_fence_after();
          b_done = true;
#pragma unroll
          for (int c = 0; c < kD; c += 32) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c, o);
            ptx::tmem_wait_ld32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            ptx::tmem_st32(tO + c, o);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sm_a);
        // second half
        if (!b_done) {
          ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(p_free_b, (nblk - 1u) & 1u, wc, 34));
          if (!ok) break;
          ptx::tc_fence_after();
        }
        p_piece(64);
        p_piece(96);
        le += se.x + se.y;
        l += sr0 + sr1;
        ptx::tmem_wait_st();
      }
      if (!ok) break;
      // the second half of the tile's last P is stored
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sm_b);
      // epilogue: O = acc / l, LSE = m + ln(le)
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(o_full, o_ph, wc, 31));
      if (!ok) break;
      o_ph ^= 1u;
      ptx::tc_fence_after();
      // this thread's row of the unnormalised O
      float oacc[kD];
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c, o);
        ptx::tmem_wait_ld32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) oacc[c + i] = __uint_as_float(o[i]);
      }
      const int prow = t * kBM + wq * 32 + lane;  // row within the pair
      // Hands the piece to the epilogue helper: this warp's writes (O rows in the Q buffer, or
      // the partial in global memory) are ordered before the arrival.
      auto release_q = [&](bool store) {
        if (store) ptx::fence_proxy_async_smem();  // shared-memory writes -> the TMA engine
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->epi[qb][t]));
      };
      if (ti.kind == 2) {
        // later blocks of a split pair: hand (O, m, l, le) to the CTA that holds its first block.
        // Column-major, so a warp's 32 rows of one column are one contiguous 128-byte line.
        float* slot = ws + static_cast<size_t>(blockIdx.x) * kSlotFloats;
#pragma unroll
        for (int c = 0; c < kD; ++c) slot[c * kPairRows + prow] = oacc[c];
        slot[kPairRows * kD + prow] = m2;
        slot[kPairRows * kD + kPairRows + prow] = l;
        slot[kPairRows * kD + 2 * kPairRows + prow] = le;
        release_q(false);  // the helper publishes the partial
        ptx::tc_fence_before();
        continue;
      }
      if (ti.kind == 1) {
        // first blocks of a split pair: merge the partials of the CTAs that took the rest
        // (they processed those pieces first, so they are normally long ready)
        const uint32_t units = Schedule<CAUSAL>::total_units(BH, num_pairs, nkb);
        const uint32_t end_u = static_cast<uint32_t>(ti.bh) * units_before<CAUSAL>(num_pairs, nkb) +
                               units_before<CAUSAL>(ti.q0 / (2 * kBM) + 1, nkb);  // the pair's last unit + 1
        for (uint32_t c2 = blockIdx.x + 1; c2 < gridDim.x && Schedule<CAUSAL>::start(bnd, c2, units) < end_u && ok;
             ++c2) {
          // a CTA with an empty range writes no partial
          if (Schedule<CAUSAL>::start(bnd, c2 + 1, units) == Schedule<CAUSAL>::start(bnd, c2, units)) continue;
          uint32_t* f = flags + static_cast<size_t>(c2) * 8 + warp;
          bool got = true;
          if (lane == 0) {
            const uint64_t t0 = ptx::globaltimer_ns();
            got = false;
            for (uint32_t k = 0; k < (1u << 30); ++k) {
              if (ptx::ld_acquire_u32(f) == epoch) {
                got = true;
                break;
              }
              if ((k & 255u) == 255u && (*wc.abort_flag || ptx::globaltimer_ns() - t0 > wc.budget_ns)) break;
            }
            if (!got) ptx::raise_error(wc, kStatusTimeout, 36);
          }
          ok = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!ok) break;
          (void)ptx::ld_acquire_u32(f);  // orders this lane's reads of the slot after the flag
          if (lane == 0) *f = 0u;          // consumed: the workspace goes back to zeros
          const float* slot = ws + static_cast<size_t>(c2) * kSlotFloats;
          const float m_p = slot[kPairRows * kD + prow];
          const float l_p = slot[kPairRows * kD + kPairRows + prow];
          const float le_p = slot[kPairRows * kD + 2 * kPairRows + prow];
          const float mn = fmaxf(m2, m_p);
          const float a = ptx::ex2(m2 - mn), b = ptx::ex2(m_p - mn);
#pragma unroll
          for (int c = 0; c < kD; ++c) oacc[c] = oacc[c] * a + slot[c * kPairRows + prow] * b;
          l = l * a + l_p * b;
          le = le * a + le_p * b;
          m2 = mn;
        }
        if (!ok) break;
      }
      // O = acc / l into the tile's Q buffer (its last S has completed before O was final) in the
      // tensor map's 128-byte swizzled layout, then one TMA store per tile (rows past M are
      // clipped by the tensor map)
      const float inv = 1.f / l;
      {
        const int r = wq * 32 + lane;  // row within the tile
        uint8_t* buf = smem_raw + (q_addr(qb, t) - raw_u32);
#pragma unroll
        for (int v = 0; v < kD / 8; ++v) {
          uint32_t h[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float a = oacc[8 * v + 2 * i] * inv, b = oacc[8 * v + 2 * i + 1] * inv;
            h[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
          }
          *reinterpret_cast<uint4*>(buf + r * 128 + ((v ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      if (row < M && LSE != nullptr) LSE[static_cast<size_t>(ti.bh) * M + row] = (m2 + __log2f(le)) * kLn2;
      release_q(true);
      // O_t is read: the next pair's first P V may overwrite it (ordered by the next sm_a arrive)
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <bool BF16, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo, float* LSE,
                     int BH, int M, int N, float scale, const FwdSplit& sp, const LaunchCtx& ctx) {
  auto kern = fwd_d64_kernel<BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>((M + 2 * kBM - 1) / (2 * kBM)) * BH;
  // Both schedules launch as programmatic dependents of the kernel before them on the stream:
  // their set-up overlaps its tail, and they touch global memory only after griddepcontrol.wait.
  // (A cooperative launch, which would guarantee the split schedule's CTAs are resident at once,
  // measured to serialise with the previous kernel, 65.5 against 62.9 us back to back at
  // B4 H12 N2048; the split schedule's one CTA per SM becomes resident as the SMs free up.)
  const SplitBounds bounds = sp.ws != nullptr ? split_bounds<CAUSAL>(BH, M, N, ctx.num_sms) : SplitBounds{};
  if (sp.ws != nullptr) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ctx.num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, LSE, BH, M, N, scale * kLog2e, sp.ws, sp.flags, sp.epoch,
                              ctx.status, ctx.wait_budget_ns, ctx.inject, bounds);
  }
  const int grid = static_cast<int>(tiles < ctx.num_sms ? tiles : ctx.num_sms);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, LSE, BH, M, N, scale * kLog2e, static_cast<float*>(nullptr),
                            static_cast<uint32_t*>(nullptr), 0u, ctx.status, ctx.wait_budget_ns, ctx.inject,
                            bounds);
}

}  // namespace

size_t fwd_d64_split_bytes(int num_sms) {
  return static_cast<size_t>(num_sms) * (kSlotFloats * sizeof(float) + 8 * sizeof(uint32_t));
}

cudaError_t launch_fwd_d64(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                           float scale, bool causal, int dtype, const FwdSplit& sp, const LaunchCtx& ctx) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_tmap_3d(&mq, Q, dtype, kD, M, BH, 64, kBM) || !make_tmap_3d(&mk, K, dtype, kD, N, BH, 64, kBN) ||
      !make_tmap_3d(&mv, V, dtype, kD, N, BH, 64, kBN) || !make_tmap_3d(&mo, O, dtype, kD, M, BH, 64, kBM))
    return cudaErrorInvalidValue;
  const bool bf = dtype == kBF16;
  if (bf) return causal ? launch_t<true, true>(mq, mk, mv, mo, LSE, BH, M, N, scale, sp, ctx)
                        : launch_t<true, false>(mq, mk, mv, mo, LSE, BH, M, N, scale, sp, ctx);
  return causal ? launch_t<false, true>(mq, mk, mv, mo, LSE, BH, M, N, scale, sp, ctx)
                : launch_t<false, false>(mq, mk, mv, mo, LSE, BH, M, N, scale, sp, ctx);
}

}  // namespace fa
