// FP8 forward prefill, head dimension 64 ("Flash Attention" notes, section "FlashAttention 3",
// the FP8 bullets): both products on E4M3 operands (tcgen05 kind::f8f6f4, f32 accumulation).
//
// The operands come from fp8_quant.cu: Q8 and K8 are Q M and K M (M the Hadamard-times-sign
// matrix, so Q8 K8^T approximates Q K^T) with one scale per 128-row block (sq, sk); Vt8 is V
// with one scale per head (sv), stored [d][keys] so that it is the K-major operand of P V.
// The schedule and the roles are those of the fp16/bf16 D = 64 forward (whole pairs of
// 128-row query tiles per CTA, one CTA per SM):
//
//   S0 [0,128)  S1 [128,256)  P0 [256,288)  P1 [288,320)  O0 [320,400)  O1 [400,480)
//
// with the softmax's exponent constant per key block j: scale * log2(e) * sq * sk[j], and the
// weights rounded to E4M3 (four per tensor-memory column) for P V. Each stage's V tile carries
// 16 constant rows after its 64 (row 64 all ones, the rest zero), so P V has N = 80 and its
// column 64 accumulates the sum of the rounded weights in the tensor core, rescaled with O;
// O is divided by that sum and multiplied by sv. LSE uses the exact f32 sum.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "fwd_common.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using fwdc::classic_tile;
using fwdc::fadd2;
using fwdc::ffma2;
using fwdc::fmax3;
using fwdc::kBM;
using fwdc::kBN;
using fwdc::mask32;
using fwdc::tile_info;
using fwdc::TileInfo;

constexpr int kD = 64;
constexpr int kQSlot = 16384;  // Q8 tile (8 KB) or, after its last S, the tile's fp16 O (16 KB)
constexpr int kKTile = kBN * kD;  // 8 KB: 128 keys x 64 bytes
constexpr int kVTile = kD * kBN;  // 8 KB: 64 rows of 128 keys (what TMA loads)
constexpr int kVRows = kD + 16;   // plus a row of ones and 15 of zeros
constexpr int kVSlot = kVRows * kBN;  // 10 KB per stage
constexpr int kDO = kVRows;       // columns of an O accumulator: 64 of O, the weight sum, 15 zeros
constexpr int kStages = 4;
constexpr int kQBuf = 2;
constexpr int kThreads = 384;
constexpr int kWarpProd = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpEpi = 11;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSmemData = kQBuf * 2 * kQSlot + kStages * (kKTile + kVSlot);
constexpr int kSmemBytes = 1024 + 1024 + kSmemData;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kColS = 0, kColP = 256, kColO = 320;
static_assert(kColO + 2 * kDO <= 512, "tensor-memory plan");

struct Hdr {
  unsigned long long q_full[kQBuf], q_empty[kQBuf];
  unsigned long long epi[kQBuf][2];
  unsigned long long kv_full[kStages], kv_empty[kStages];
  unsigned long long s_full[2];
  unsigned long long sm_a[2];
  unsigned long long sm_b[2];
  unsigned long long p_free_a[2];
  unsigned long long p_free_b[2];
  unsigned long long o_full[2];
  unsigned long long mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   float* __restrict__ LSE, const float* __restrict__ sq, const float* __restrict__ sk,
                   const float* __restrict__ sv, int BH, int M, int N, float scale_log2_signed, DevStatus* status,
                   unsigned long long budget_ns) {
  extern __shared__ uint8_t smem_raw[];
  Hdr* hdr = reinterpret_cast<Hdr*>(smem_raw);
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t data_u32 = (raw_u32 + 1024u + 1023u) & ~1023u;
  auto q_addr = [&](int qb, int t) { return data_u32 + (qb * 2 + t) * kQSlot; };
  auto k_addr = [&](int st) { return data_u32 + kQBuf * 2 * kQSlot + st * (kKTile + kVSlot); };
  auto v_addr = [&](int st) { return k_addr(st) + kKTile; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_pairs = (M + 2 * kBM - 1) / (2 * kBM);
  const int nkb = (N + kBN - 1) / kBN;
  const int nqb = (M + kBM - 1) / kBM;
  const int num_tiles = num_pairs * BH;
  // scale < 0: the score product is negated in the tensor core and the softmax scales by |scale|
  // (kept above 1e-30 so that masked scores stay -inf when scale = 0)
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
  // the constant rows of every stage's V tile: row 64 all E4M3 ones (0x38), rows 65..79 zero
  // (each row's 16-byte chunks are equal, so the 128-byte swizzle leaves them in place)
  for (int i = threadIdx.x; i < kStages * (kVSlot - kVTile) / 16; i += kThreads) {
    const int st = i / ((kVSlot - kVTile) / 16), c = i % ((kVSlot - kVTile) / 16);
    const uint32_t w = c < kBN / 16 ? 0x38383838u : 0u;
    *reinterpret_cast<uint4*>(smem_raw + (v_addr(st) - raw_u32) + kVTile + 16 * c) = make_uint4(w, w, w, w);
  }
  ptx::fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's reads
  if (warp == kWarpProd && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  if (warp == kWarpEpi && lane == 0) ptx::prefetch_tmap(&tmO);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  ptx::WaitCtx wc{&hdr->abort_flag, status, budget_ns, kKernFwdFp8};
  // launched as a programmatic dependent: the set-up above overlapped the previous kernel's tail;
  // no global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_it = 0;
      bool ok = true;
      int it = 0;  // pieces taken; one Q load each
      for (; ok; ++it) {
        const int tile = classic_tile<CAUSAL>(it);
        if (tile >= num_tiles) break;
        const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
        const int qb = it % kQBuf;
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->q_empty[qb]), (static_cast<uint32_t>(it / kQBuf) & 1u) ^ 1u, wc, 10))
          break;
        const uint32_t qf = ptx::smem_u32(&hdr->q_full[qb]);
        ptx::mbar_arrive_expect_tx(qf, 2 * kBM * kD);
        for (int t = 0; t < 2; ++t) ptx::tma_load_3d(q_addr(qb, t), &tmQ, qf, 0, ti.q0 + t * kBM, ti.bh);
        for (int j = 0; j < ti.nb1; ++j, ++kv_it) {
          const int st = kv_it % kStages;
          if (!ptx::mbar_wait(ptx::smem_u32(&hdr->kv_empty[st]), ((kv_it / kStages) & 1u) ^ 1u, wc, 11)) {
            ok = false;
            break;
          }
          const uint32_t f = ptx::smem_u32(&hdr->kv_full[st]);
          ptx::mbar_arrive_expect_tx(f, kKTile + kVTile);
          ptx::tma_load_3d(k_addr(st), &tmK, f, 0, j * kBN, ti.bh);
          ptx::tma_load_3d(v_addr(st), &tmV, f, j * kBN, 0, ti.bh);
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = kv_it > (uint32_t)kStages ? kv_it - kStages : 0u; k < kv_it; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->kv_full[k % kStages]), (k / kStages) & 1u, 100000000ull);
        for (int k = it > kQBuf ? it - kQBuf : 0; k < it; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->q_full[k % kQBuf]), static_cast<uint32_t>(k / kQBuf) & 1u, 100000000ull);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpMma + 1) {
    // ------------------------------------------------------------ MMA issuer of tile t (lane 0)
    const uint32_t idesc_qk =
        ptx::idesc_f32acc(kBM, kBN, ptx::kFmtE4M3, ptx::kFmtE4M3, false, false) | (neg_scale ? ptx::kNegateA : 0u);
    constexpr uint32_t idesc_pv = ptx::idesc_f32acc(kBM, kDO, ptx::kFmtE4M3, ptx::kFmtE4M3, false, false);
    const int t = warp - kWarpMma;
    if (lane == 0) {
      uint32_t kv_base = 0;
      uint32_t n_a = 0, n_b = 0;
      bool ok = true;
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      const uint32_t dS = tmem + kColS + t * kBN;
      const uint32_t dO = tmem + kColO + t * kDO;
      const uint32_t aP = tmem + kColP + t * (kBN / 4);
      for (int it = 0; ok; ++it) {
        const int tile = classic_tile<CAUSAL>(it);
        if (tile >= num_tiles) break;
        const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
        const int qb = it % kQBuf;
        const int nb = t == 0 ? ti.nb0 : ti.nb1;
        if (!wait(&hdr->q_full[qb], static_cast<uint32_t>(it / kQBuf) & 1u, 20)) break;
        auto kv_ready = [&](int j) {
          const uint32_t kv = kv_base + j;
          return wait(&hdr->kv_full[kv % kStages], (kv / kStages) & 1u, 21);
        };
        auto arrival_a = [&]() { return wait(&hdr->sm_a[t], (n_a++) & 1u, 22); };
        auto arrival_b = [&]() { return wait(&hdr->sm_b[t], (n_b++) & 1u, 23); };
        // S_t(j) = Q8_t K8_j^T: two K = 32 steps over the 64-byte rows (64-byte swizzle)
        auto qk = [&](int j) {
          ptx::tc_fence_after();
          const uint64_t a0 = ptx::sdesc_sw64(q_addr(qb, t), 16, 512);
          const uint64_t b0 = ptx::sdesc_sw64(k_addr((kv_base + j) % kStages), 16, 512);
#pragma unroll
          for (int ks = 0; ks < kD / 32; ++ks) ptx::mma_f8_ss(dS, a0 + 2 * ks, b0 + 2 * ks, idesc_qk, ks > 0 ? 1u : 0u);
          commit(&hdr->s_full[t]);
        };
        // O_t (+)= P_t(j) V_j over keys [64h, 64h + 64): A from tensor memory (8 columns per 32
        // keys), B the [d][keys] tile read K-major (128-byte swizzle, 32 keys per step)
        auto pv = [&](int j, int h) {
          ptx::tc_fence_after();
          const uint64_t b0 = ptx::sdesc_sw128(v_addr((kv_base + j) % kStages), 16, 1024);
#pragma unroll
          for (int ks = 2 * h; ks < 2 * h + 2; ++ks)
            ptx::mma_f8_ts(dO, aP + ks * 8, b0 + 2 * ks, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          commit(h == 0 ? &hdr->p_free_a[t] : &hdr->p_free_b[t]);
          if (h == 1 && j == nb - 1) commit(&hdr->o_full[t]);
        };
        ok = kv_ready(0);
        if (ok) qk(0);
        if (ok && nb > 1) {
          ok = arrival_b() && kv_ready(1);
          if (ok) qk(1);
        }
        for (int j = 0; j < nb && ok; ++j) {
          if (j + 2 < nb) {
            ok = kv_ready(j + 2);
            if (!ok) break;
          }
          ok = arrival_a();
          if (!ok) break;
          pv(j, 0);
          ok = arrival_b();
          if (!ok) break;
          pv(j, 1);
          if (j + 2 < nb) qk(j + 2);
          commit(&hdr->kv_empty[(kv_base + j) % kStages]);
        }
        for (int j = nb; j < ti.nb1 && ok; ++j) {
          ok = kv_ready(j);
          if (ok) commit(&hdr->kv_empty[(kv_base + j) % kStages]);
        }
        kv_base += ti.nb1;
      }
      commit(&hdr->mma_done[t]);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done[t]), 0u, 1000000000ull);
    }
  } else if (warp == kWarpEpi) {
    // ------------------------------------------------------------ epilogue helper (lane 0)
    if (lane == 0) {
      for (int it = 0;; ++it) {
        const int tile = classic_tile<CAUSAL>(it);
        if (tile >= num_tiles) break;
        const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
        const int qb = it % kQBuf;
        const uint32_t ph = static_cast<uint32_t>(it / kQBuf) & 1u;
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t) {
          ok = ptx::mbar_wait(ptx::smem_u32(&hdr->epi[qb][t]), ph, wc, 37);
          if (ok) {
            ptx::tma_store_3d(&tmO, q_addr(qb, t), 0, ti.q0 + t * kBM, ti.bh);
            ptx::bulk_commit();
          }
        }
        if (!ok) break;
        ptx::bulk_wait_read();
        ptx::mbar_arrive(ptx::smem_u32(&hdr->q_empty[qb]));
      }
      ptx::bulk_wait_all();
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (one row per thread)
    const int t = warp >> 2;
    const int wq = warp & 3;
    const uint32_t lane_sel = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_sel + kColS + t * kBN;
    const uint32_t tP = tmem + lane_sel + kColP + t * (kBN / 4);
    const uint32_t tO = tmem + lane_sel + kColO + t * kDO;
    const uint32_t s_full = ptx::smem_u32(&hdr->s_full[t]);
    const uint32_t sm_a = ptx::smem_u32(&hdr->sm_a[t]);
    const uint32_t sm_b = ptx::smem_u32(&hdr->sm_b[t]);
    const uint32_t p_free_a = ptx::smem_u32(&hdr->p_free_a[t]);
    const uint32_t p_free_b = ptx::smem_u32(&hdr->p_free_b[t]);
    const uint32_t o_full = ptx::smem_u32(&hdr->o_full[t]);
    uint32_t nblk = 0u;
    uint32_t o_ph = 0u;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int tile = classic_tile<CAUSAL>(it);
      if (tile >= num_tiles) break;
      const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
      const int nbt = t == 0 ? ti.nb0 : ti.nb1;
      const int qb = it % kQBuf;
      const int row = ti.q0 + t * kBM + wq * 32 + lane;
      // this tile's Q scale times scale * log2(e); the key block's scale joins per block
      const int qtile = (ti.q0 + t * kBM) / kBM;
      const float csq = scale_log2 * (qtile < nqb ? sq[static_cast<size_t>(ti.bh) * nqb + qtile] : 1.f);
      const float* skh = sk + static_cast<size_t>(ti.bh) * nkb;
      float m2 = -INFINITY;
      float le = 0.f;
      for (int j = 0; j < nbt; ++j, ++nblk) {
        const float cj = csq * __ldg(skh + j);
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(s_full, nblk & 1u, wc, 30));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t r[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) ptx::tmem_ld32(tS + c, r + c);
#pragma unroll
        for (int c = 0; c < kBN; c += 32) ptx::tmem_wait_ld32(r + c);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && (j > 0 || nbt > 1)) ptx::mbar_arrive(sm_b);

        const int kbase = j * kBN;
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
        const float mxs = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cj;
        const bool rescale = j == 0 || __any_sync(0xFFFFFFFFu, mxs > m2 + kRescaleThreshold);
        float corr = 1.f;
        if (rescale) {
          const float m_new = fmaxf(m2, mxs);
          corr = m_new == -INFINITY ? 1.f : ptx::ex2(m2 - m_new);
          le *= corr;
          m2 = m_new;
        }
        const float neg_m = m2 == -INFINITY ? 0.f : -m2;
        const float2 c2 = make_float2(cj, cj), nm2 = make_float2(neg_m, neg_m);
        float2 se = make_float2(0.f, 0.f);
        // P over keys [c, c + 32): E4M3, four per column, stored to columns [c/4, c/4 + 8)
        auto p_piece = [&](int c) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t hw[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int k = c + 4 * i + 2 * u;
              const float2 x = ffma2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), c2, nm2);
              const float a = ptx::ex2(x.x), b = ptx::ex2(x.y);
              se = fadd2(se, make_float2(a, b));
              hw[u] = ptx::pack_e4m3x2(a, b);
            }
            pk[i] = hw[0] | (hw[1] << 16);
          }
          ptx::tmem_st8(tP + c / 4, pk);
        };
        if (nblk > 0u) {
          ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(p_free_a, (nblk - 1u) & 1u, wc, 32));
          if (!ok) break;
          ptx::tc_fence_after();
        }
        p_piece(0);
        p_piece(32);
        bool b_done = nblk == 0u;
        if (rescale && j > 0) {
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
          {  // the weight sum (column 64) with it
            uint32_t o[16];
            ptx::tmem_ld16(tO + kD, o);
            ptx::tmem_wait_ld16(o);
            o[0] = __float_as_uint(__uint_as_float(o[0]) * corr);
            ptx::tmem_st16(tO + kD, o);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sm_a);
        if (!b_done) {
          ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(p_free_b, (nblk - 1u) & 1u, wc, 34));
          if (!ok) break;
          ptx::tc_fence_after();
        }
        p_piece(64);
        p_piece(96);
        le += se.x + se.y;
        ptx::tmem_wait_st();
      }
      if (!ok) break;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sm_b);
      ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(o_full, o_ph, wc, 31));
      if (!ok) break;
      o_ph ^= 1u;
      ptx::tc_fence_after();
      // O = acc * sv / l, into the tile's Q slot in the 128-byte swizzled layout of the O map
      float l;
      {
        uint32_t o[16];
        ptx::tmem_ld16(tO + kD, o);
        ptx::tmem_wait_ld16(o);
        l = __uint_as_float(o[0]);  // the sum of the rounded weights, from the tensor core
      }
      const float f = sv[ti.bh] / l;
      const int r_in = wq * 32 + lane;
      uint8_t* buf = smem_raw + (q_addr(qb, t) - raw_u32);
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c, o);
        ptx::tmem_wait_ld32(o);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t h[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float a = __uint_as_float(o[8 * v + 2 * i]) * f, b = __uint_as_float(o[8 * v + 2 * i + 1]) * f;
            h[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
          }
          const int chunk = c / 8 + v;
          *reinterpret_cast<uint4*>(buf + r_in * 128 + ((chunk ^ (r_in & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      if (row < M && LSE != nullptr) LSE[static_cast<size_t>(ti.bh) * M + row] = (m2 + __log2f(le)) * kLn2;
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&hdr->epi[qb][t]));
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
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                     float* LSE, const Fp8Ws& w, int BH, int M, int N, float scale, const LaunchCtx& ctx) {
  auto kern = fwd_fp8_kernel<BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>((M + 2 * kBM - 1) / (2 * kBM)) * BH;
  const int grid = static_cast<int>(tiles < ctx.num_sms ? tiles : ctx.num_sms);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];  // a programmatic dependent of the kernel before it on the stream
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, LSE, static_cast<const float*>(w.sq), static_cast<const float*>(w.sk),
                            static_cast<const float*>(w.sv), BH, M, N, scale * kLog2e, ctx.status, ctx.wait_budget_ns);
}

}  // namespace

cudaError_t launch_fwd_fp8(const Fp8Ws& w, void* O, float* LSE, int BH, int M, int N, float scale, bool causal,
                           int dtype, const LaunchCtx& ctx) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_tmap_3d_ex(&mq, w.q8, kU8, kD, M, BH, kD, kBM, 64) ||
      !make_tmap_3d_ex(&mk, w.k8, kU8, kD, N, BH, kD, kBN, 64) ||
      !make_tmap_3d_ex(&mv, w.vt8, kU8, w.npad, kD, BH, kBN, kD, 128) ||
      !make_tmap_3d(&mo, O, dtype, kD, M, BH, 64, kBM))
    return cudaErrorInvalidValue;
  const bool bf = dtype == kBF16;
  if (bf) return causal ? launch_t<true, true>(mq, mk, mv, mo, LSE, w, BH, M, N, scale, ctx)
                        : launch_t<true, false>(mq, mk, mv, mo, LSE, w, BH, M, N, scale, ctx);
  return causal ? launch_t<false, true>(mq, mk, mv, mo, LSE, w, BH, M, N, scale, ctx)
                : launch_t<false, false>(mq, mk, mv, mo, LSE, w, BH, M, N, scale, ctx);
}

}  // namespace fa
