// Forward prefill for fp16 / bf16 inputs on tcgen05 tensor cores.
//
// The method is FlashAttention-2's forward ("Flash attention, f32", Phobos
// examples: one block of query rows per CTA, a running max m, denominator l and
// unnormalised accumulator carried across key blocks, one division at the end;
// "06: Fused attention": the causal walk that stops at the diagonal and the
// stored statistic L = m + log l; "Flash Attention" notes, FlashAttention 4:
// single-thread tcgen05 issue, S/P/O in tensor memory, conditional rescaling).
//
// GB300 layout of the work:
//  * a CTA owns a pair of 128-row query tiles of one (batch, head) and runs
//    persistently over such pairs (non-causal: the pairs of a head are adjacent
//    so resident CTAs share that head's K/V in L2; causal: heaviest pairs first);
//  * warp 8 issues TMA loads: both Q tiles once per pair, then K and V blocks
//    of 128 keys into a ring of shared-memory stages (128-byte swizzle);
//  * warp 9 (one thread) issues the MMAs: S_t = Q_t K^T into tensor memory,
//    O_t += P_t V with P_t read from tensor memory;
//  * warps 0-3 and 4-7 are the softmax of tile 0 and tile 1: each thread owns
//    one query row (one TMEM lane). The two tiles ping-pong so one tile's
//    softmax overlaps the other tile's MMAs.
//
// Softmax of one key block, per row. The running maximum is kept stale unless
// the block's maximum exceeds it by more than 2^8 (base-2 units), the FA4
// conditional rescale; O and l share the stale maximum so the result is exact.
// Speculative single pass: the scores are read once, P = 2^(s*c - m) is formed
// against the current maximum while the block maximum is tracked; only when
// that maximum breaks the threshold (always on the first block) are the scores
// read again with the new maximum and O rescaled in tensor memory. P stays in
// registers until the decision, then is written as packed halves over the
// scores' first 64 columns.
//
// O is divided by the sum of the half-rounded weights that multiplied V, so it
// is a weighted mean of V rows (that sum is formed in registers); LSE uses the
// exact f32 sum.
//
// This file serves D = 128; D = 64 has its own kernel (fwd_d64.cu), whose
// tensor-memory plan only fits when D = 64.
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "fwd_common.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using fwdc::kBM;
using fwdc::kBN;
using fwdc::TileInfo;
using fwdc::tile_info;
using fwdc::ffma2;
using fwdc::fadd2;
using fwdc::fmax3;
using fwdc::classic_tile;
using fwdc::mask32;
constexpr int kChunk = 16384;   // one 128-row x 128-byte swizzled chunk
// 10 warps: three share one SM sub-partition (16K registers), so a thread has
// at most 168 registers.
constexpr int kThreads = 320;   // 8 softmax warps + producer + MMA
constexpr int kWarpProd = 8;
constexpr int kWarpMma = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  static_assert(D == 128, "this kernel serves D = 128");
  static constexpr int kDC = D / 64;                       // 64-column chunks
  static constexpr int kTileBytes = kDC * kChunk;          // one Q tile / K block / V block
  static constexpr int kStages = 2;                        // K/V ring depth
  static constexpr int kQBuf = 1;                          // Q pair buffers
  static constexpr int kDO = D;                            // O columns in tensor memory
  static constexpr int kSmemData = kQBuf * 2 * kTileBytes + kStages * 2 * kTileBytes;
  static constexpr int kSmemBytes = 1024 + 1024 + kSmemData;  // header + alignment slack + data
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct FwdHdr {
  unsigned long long q_full[2], q_empty[2];
  unsigned long long k_full[4], v_full[4], kv_empty[4];
  unsigned long long s_full[2], p_full[2], o_full[2];
  unsigned long long mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// P for 32 scores against the current maximum: packed halves into pk[16],
// exact sum into se, rounded sum into sr (only when ROUNDED), and the raw
// maximum into mx.
template <bool BF16, bool ROUNDED>
__device__ __forceinline__ void p_chunk(const uint32_t* r, float sl2, float neg_m, float& mx, float2& se, float2& sr,
                                        uint32_t* pk) {
  const float2 c2 = make_float2(sl2, sl2), m2 = make_float2(neg_m, neg_m);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 s = make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    mx = fmax3(mx, s.x, s.y);
    const float2 x = ffma2(s, c2, m2);
    const float a = ptx::ex2(x.x), b = ptx::ex2(x.y);
    se = fadd2(se, make_float2(a, b));
    pk[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
    if (ROUNDED) sr = fadd2(sr, BF16 ? ptx::unpack_bf16x2(pk[i]) : ptx::unpack_f16x2(pk[i]));
  }
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_half_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, void* __restrict__ Optr, float* __restrict__ LSE,
                    int BH, int M, int N, float scale_log2_signed, DevStatus* status, unsigned long long budget_ns) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  FwdHdr* hdr = reinterpret_cast<FwdHdr*>(smem_raw);
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t data_u32 = (raw_u32 + 1024u + 1023u) & ~1023u;  // 1024-aligned for the swizzle atoms
  // data layout: Q[qbuf][tile], then stages (K, V)
  auto q_addr = [&](int qb, int t) { return data_u32 + (qb * 2 + t) * C::kTileBytes; };
  auto k_addr = [&](int st) { return data_u32 + C::kQBuf * 2 * C::kTileBytes + st * 2 * C::kTileBytes; };
  auto v_addr = [&](int st) { return k_addr(st) + C::kTileBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_pairs = (M + 2 * kBM - 1) / (2 * kBM);
  const int nkb = (N + kBN - 1) / kBN;
  const int num_tiles = num_pairs * BH;
  // scale < 0: the score product is negated in the tensor core and the softmax scales by |scale|.
  // |scale| is kept above 1e-30 so that a masked score (-inf) times it stays -inf when scale = 0
  // (every visible weight is then exp2 of about 0, i.e. 1).
  const bool neg_scale = scale_log2_signed < 0.f;
  const float scale_log2 = fmaxf(fabsf(scale_log2_signed), 1e-30f);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&hdr->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->q_empty[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->p_full[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&hdr->o_full[i]), 1);
    }
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(ptx::smem_u32(&hdr->k_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->v_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&hdr->kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&hdr->mma_done), 1);
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
  }
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
      int it = 0;
      bool ok = true;
      for (int r = 0, tile = classic_tile<CAUSAL>(0); tile < num_tiles && ok; tile = classic_tile<CAUSAL>(++r), ++it) {
        const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
        const int qb = it % C::kQBuf;
        const uint32_t qph = static_cast<uint32_t>(it / C::kQBuf) & 1u;
        if (!ptx::mbar_wait(ptx::smem_u32(&hdr->q_empty[qb]), qph ^ 1u, wc, 10)) break;
        const uint32_t qf = ptx::smem_u32(&hdr->q_full[qb]);
        ptx::mbar_arrive_expect_tx(qf, 2 * C::kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < C::kDC; ++c)
            ptx::tma_load_3d(q_addr(qb, t) + c * kChunk, &tmQ, qf, c * 64, ti.q0 + t * kBM, ti.bh);
        const int nb = ti.nb1;
        for (int j = 0; j < nb; ++j, ++kv_it) {
          const int st = kv_it % C::kStages;
          const uint32_t ph = (kv_it / C::kStages) & 1u;
          if (!ptx::mbar_wait(ptx::smem_u32(&hdr->kv_empty[st]), ph ^ 1u, wc, 11)) {
            ok = false;
            break;
          }
          const uint32_t kf = ptx::smem_u32(&hdr->k_full[st]);
          ptx::mbar_arrive_expect_tx(kf, C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) ptx::tma_load_3d(k_addr(st) + c * kChunk, &tmK, kf, c * 64, j * kBN, ti.bh);
          const uint32_t vf = ptx::smem_u32(&hdr->v_full[st]);
          ptx::mbar_arrive_expect_tx(vf, C::kTileBytes);
          for (int c = 0; c < C::kDC; ++c) ptx::tma_load_3d(v_addr(st) + c * kChunk, &tmV, vf, c * 64, j * kBN, ti.bh);
        }
      }
      if (hdr->abort_flag) {  // let issued copies land before shared memory is released
        for (uint32_t k = kv_it > (uint32_t)C::kStages ? kv_it - C::kStages : 0u; k < kv_it; ++k) {
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->k_full[k % C::kStages]), (k / C::kStages) & 1u, 100000000ull);
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->v_full[k % C::kStages]), (k / C::kStages) & 1u, 100000000ull);
        }
        // Q loads issued: one per piece taken (it)
        for (int k = it > C::kQBuf ? it - C::kQBuf : 0; k < it; ++k)
          ptx::mbar_wait_drain(ptx::smem_u32(&hdr->q_full[k % C::kQBuf]), static_cast<uint32_t>(k / C::kQBuf) & 1u,
                               100000000ull);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 alone runs this role. One issuer serves both tiles in the order
    // PV_{0,j-1}, QK_{0,j}, PV_{1,j-1}, QK_{1,j}: a tcgen05.mma issue blocks while the
    // tensor pipe is busy, so each tile's group runs back to back (measured faster
    // than one issuer per tile, whose MMAs interleave in the pipe, and than a
    // warp-wide loop).
    constexpr uint32_t fmt = BF16 ? ptx::kFmtBF16 : ptx::kFmtF16;
    const uint32_t idesc_qk = ptx::idesc_f32acc(kBM, kBN, fmt, fmt, false, false) | (neg_scale ? ptx::kNegateA : 0u);
    constexpr uint32_t idesc_pv = ptx::idesc_f32acc(kBM, C::kDO, fmt, fmt, false, true);
    if (lane == 0) {
      uint32_t kv_it = 0;
      uint32_t p_ph[2] = {0u, 0u};
      int it = 0;
      bool ok = true;
      // descriptor of a byte offset from a descriptor: the start address field is addr >> 4
      auto qk = [&](int t, int qb, int st) {
        const uint64_t a0 = ptx::sdesc_sw128(q_addr(qb, t), 16, 1024);
        const uint64_t b0 = ptx::sdesc_sw128(k_addr(st), 16, 1024);
        const uint32_t d = tmem + t * kBN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t off = static_cast<uint64_t>(((ks >> 2) * kChunk + (ks & 3) * 32) >> 4);
          ptx::mma_f16_ss(d, a0 + off, b0 + off, idesc_qk, ks > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](int t, int st, bool accumulate) {
        // the second 64-column group of B is the next V chunk
        const uint32_t lbo = kChunk;
        const uint64_t b0 = ptx::sdesc_sw128(v_addr(st), lbo, 1024);
        const uint32_t d = tmem + 2 * kBN + t * 128;
        const uint32_t p = tmem + t * kBN;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          ptx::mma_f16_ts(d, p + ks * 8, b0 + static_cast<uint64_t>((ks * 2048) >> 4), idesc_pv,
                          (accumulate || ks > 0) ? 1u : 0u);
      };
      auto commit = [&](unsigned long long* bar) { ptx::tc_commit(ptx::smem_u32(bar)); };
      auto wait = [&](unsigned long long* bar, uint32_t parity, uint32_t site) {
        return ptx::mbar_wait(ptx::smem_u32(bar), parity, wc, site);
      };
      for (int r = 0, tile = classic_tile<CAUSAL>(0); tile < num_tiles && ok; tile = classic_tile<CAUSAL>(++r), ++it) {
        const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
        const int qb = it % C::kQBuf;
        const uint32_t qph = static_cast<uint32_t>(it / C::kQBuf) & 1u;
        if (!wait(&hdr->q_full[qb], qph, 20)) break;
        ptx::tc_fence_after();
        const int nb = ti.nb1;
        for (int j = 0; j <= nb && ok; ++j) {
          const uint32_t cur = kv_it + j, prev = kv_it + j - 1;
          const int st = cur % C::kStages, pst = prev % C::kStages;
          if (j < nb) {
            ok = wait(&hdr->k_full[st], (cur / C::kStages) & 1u, 21);
            if (!ok) break;
            ptx::tc_fence_after();
          }
          if (j >= 1 && j - 1 < ti.nb0) {
            ok = wait(&hdr->p_full[0], p_ph[0], 22) && wait(&hdr->v_full[pst], (prev / C::kStages) & 1u, 23);
            if (!ok) break;
            p_ph[0] ^= 1u;
            ptx::tc_fence_after();
            pv(0, pst, j - 1 > 0);
            if (j - 1 == ti.nb0 - 1) commit(&hdr->o_full[0]);
          }
          if (j < ti.nb0) {
            qk(0, qb, st);
            commit(&hdr->s_full[0]);
          }
          if (j >= 1) {
            ok = wait(&hdr->p_full[1], p_ph[1], 24) && wait(&hdr->v_full[pst], (prev / C::kStages) & 1u, 25);
            if (!ok) break;
            p_ph[1] ^= 1u;
            ptx::tc_fence_after();
            pv(1, pst, j - 1 > 0);
            if (j - 1 == nb - 1) commit(&hdr->o_full[1]);
            commit(&hdr->kv_empty[pst]);
          }
          if (j < nb) {
            qk(1, qb, st);
            commit(&hdr->s_full[1]);
            if (j == nb - 1) commit(&hdr->q_empty[qb]);
          }
        }
        kv_it += nb;
      }
      // every MMA issued by lane 0 has completed once mma_done flips
      commit(&hdr->mma_done);
      ptx::mbar_wait_drain(ptx::smem_u32(&hdr->mma_done), 0u, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    constexpr bool kRounded = true;  // rounded row sum formed in registers
    const int t = warp >> 2;          // which tile of the pair
    const int wq = warp & 3;          // TMEM lane quarter
    const uint32_t lane_sel = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_sel + t * kBN;
    const uint32_t tO = tmem + lane_sel + 2 * kBN + t * 128;
    const uint32_t s_full = ptx::smem_u32(&hdr->s_full[t]);
    const uint32_t p_full = ptx::smem_u32(&hdr->p_full[t]);
    const uint32_t o_full = ptx::smem_u32(&hdr->o_full[t]);
    uint32_t s_ph = 0u, o_ph = 0u;
    bool ok = true;
    for (int r = 0, tile = classic_tile<CAUSAL>(0); tile < num_tiles && ok; tile = classic_tile<CAUSAL>(++r)) {
      const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
      const int nbt = t == 0 ? ti.nb0 : ti.nb1;
      const int row = ti.q0 + t * kBM + wq * 32 + lane;  // query index within the head
      float m2 = -INFINITY;  // running max of scale*log2(e)*s (possibly stale by < 2^8)
      float l = 0.f;         // sum of the half-rounded weights (D = 128 only; D = 64 reads it from O)
      float le = 0.f;        // sum of the exact f32 weights (gives LSE)
      for (int j = 0; j < nbt; ++j) {
        ok = ptx::mbar_wait(s_full, s_ph, wc, 30);
        __syncwarp();  // lanes may leave the poll at different times; reconverge for .aligned ops
        if (!ok) break;
        s_ph ^= 1u;
        ptx::tc_fence_after();
        const int kbase = j * kBN;
        const bool edge = (kbase + kBN > N) || (CAUSAL && kbase + kBN - 1 > ti.q0 + t * kBM);

        // -- speculative single pass against the current maximum
        bool slow = (j == 0);
        uint32_t pk[kBN / 2];
        float2 se = make_float2(0.f, 0.f), sr = make_float2(0.f, 0.f);
        if (!slow) {
          float mx = -INFINITY;
          const float neg_m = -m2;
          uint32_t r[2][32];
          ptx::tmem_ld32(tS, r[0]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            ptx::tmem_wait_ld32(r[c & 1]);
            if (c < 3) ptx::tmem_ld32(tS + 32 * (c + 1), r[(c + 1) & 1]);
            if (edge) mask32<CAUSAL>(r[c & 1], kbase + 32 * c, N, row);
            p_chunk<BF16, kRounded>(r[c & 1], scale_log2, neg_m, mx, se, sr, pk + 16 * c);
          }
          slow = __any_sync(0xFFFFFFFFu, mx * scale_log2 > m2 + kRescaleThreshold);
        }
        if (slow) {
          // -- block maximum first, then rescale O if the maximum moved, then P
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBN; c += 32) {
            uint32_t r[32];
            ptx::tmem_ld32(tS + c, r);
            ptx::tmem_wait_ld32(r);
            if (edge) mask32<CAUSAL>(r, kbase + c, N, row);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              mx0 = fmaxf(mx0, __uint_as_float(r[i]));
              mx1 = fmaxf(mx1, __uint_as_float(r[i + 1]));
            }
          }
          const float m_new = fmaxf(m2, fmaxf(mx0, mx1) * scale_log2);
          const float corr = m_new == -INFINITY ? 1.f : ptx::ex2(m2 - m_new);
          l *= corr;
          le *= corr;
          if (j > 0) {  // O holds earlier blocks: rescale it (the previous PV has completed)
            uint32_t o[16];
#pragma unroll
            for (int c = 0; c < C::kDO; c += 16) {
              ptx::tmem_ld16(tO + c, o);
              ptx::tmem_wait_ld16(o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
              ptx::tmem_st16(tO + c, o);
            }
          }
          m2 = m_new;
          const float neg_m = m2 == -INFINITY ? 0.f : -m2;
          float mx_unused = -INFINITY;
          se = make_float2(0.f, 0.f);
          sr = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kBN; c += 32) {
            uint32_t r[32];
            ptx::tmem_ld32(tS + c, r);
            ptx::tmem_wait_ld32(r);
            if (edge) mask32<CAUSAL>(r, kbase + c, N, row);
            p_chunk<BF16, kRounded>(r, scale_log2, neg_m, mx_unused, se, sr, pk + c / 2);
          }
        }
        le += se.x + se.y;
        if (kRounded) l += sr.x + sr.y;
        // P over the scores' first 64 columns (all scores have been read)
        ptx::tmem_st32(tS + 0, pk);
        ptx::tmem_st32(tS + 32, pk + 32);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full);
      }
      if (!ok) break;
      // epilogue: O = acc / l, LSE = m + ln l
      ok = ptx::mbar_wait(o_full, o_ph, wc, 31);
      __syncwarp();
      if (!ok) break;
      o_ph ^= 1u;
      ptx::tc_fence_after();
      const float inv = 1.f / l;
      const bool valid = row < M;
      const size_t orow = (static_cast<size_t>(ti.bh) * M + (valid ? row : 0)) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c, o);
        ptx::tmem_wait_ld32(o);
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = __uint_as_float(o[2 * i]) * inv, b = __uint_as_float(o[2 * i + 1]) * inv;
          h[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(Optr) + orow + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      if (valid && LSE != nullptr) LSE[static_cast<size_t>(ti.bh) * M + row] = (m2 + __log2f(le)) * kLn2;
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

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* O, float* LSE,
                     int BH, int M, int N, float scale, const LaunchCtx& ctx) {
  using C = FwdCfg<D>;
  auto kern = fwd_half_kernel<D, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>((M + 2 * kBM - 1) / (2 * kBM)) * BH;
  const int grid = static_cast<int>(tiles < ctx.num_sms ? tiles : ctx.num_sms);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];  // a programmatic dependent of the kernel before it on the stream
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, O, LSE, BH, M, N, scale * kLog2e, ctx.status, ctx.wait_budget_ns);
}

}  // namespace

cudaError_t launch_fwd_half(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                            int D, float scale, bool causal, int dtype, const FwdSplit& sp, const LaunchCtx& ctx) {
  if (D == 64) return launch_fwd_d64(Q, K, V, O, LSE, BH, M, N, scale, causal, dtype, sp, ctx);
  if (D != 128) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_tmap_3d(&mq, Q, dtype, D, M, BH, 64, kBM) || !make_tmap_3d(&mk, K, dtype, D, N, BH, 64, kBN) ||
      !make_tmap_3d(&mv, V, dtype, D, N, BH, 64, kBN))
    return cudaErrorInvalidValue;
  const bool bf = dtype == kBF16;
#define FA_L(DD, BB, CC) \
  if (D == DD && bf == BB && causal == CC) return launch_t<DD, BB, CC>(mq, mk, mv, O, LSE, BH, M, N, scale, ctx);
  FA_L(128, false, false)
  FA_L(128, false, true)
  FA_L(128, true, false)
  FA_L(128, true, true)
#undef FA_L
  return cudaErrorNotSupported;
}

}  // namespace fa
