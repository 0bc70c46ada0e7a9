// The split schedule of the fp16 / bf16 D = 64 forward: every SM takes a contiguous share of the
// (query pair, key block) units of all heads; a pair cut by a share boundary is finished by the
// CTA holding its first blocks, which merges the partials the CTAs holding the rest wrote into
// their workspace slots (the online-softmax rescaling between key blocks). The pieces, their
// order and the host's share boundaries live here, apart from the kernel's per-block work.
#pragma once

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "fwd_common.cuh"

namespace fa {
namespace fwds {

using fwdc::classic_tile;
using fwdc::kBM;
using fwdc::kBN;
using fwdc::tile_info;
using fwdc::TileInfo;

constexpr int kSplitD = 64;  // head dimension of the kernels that split

// Partial result of a piece (see Schedule), one slot per CTA: O (unnormalised,
// 256 rows x 64 columns), the running maximum (log2 units), the rounded and the
// exact weight sums, f32; plus one ready flag per softmax warp.
constexpr int kPairRows = 2 * kBM;
constexpr int kSlotFloats = kPairRows * kSplitD + 3 * kPairRows;

// A CTA's unit of work: tile t of pair `pair` processes key blocks [jb, jb + nb_t).
struct Piece {
  int pair, bh, q0, jb, nb0, nb1;
  int kind;  // 0: the whole pair; 1: its first blocks, finished here together with the partials of
             // the CTAs that took the rest; 2: later blocks, written out as a partial
};

// Units of the split schedule: the key blocks of a pair's tile 0, pairs of one head adjacent
// and in query order. Non-causal every pair has nkb of them. Causal, pair p's tile 0 (queries
// [256p, 256p + 128)) needs min(nkb, 2p + 1) blocks and its tile 1 one more while that is
// <= nkb (its diagonal block, taken by the piece that holds the pair's last unit), so the
// pairs before p hold p^2 units while 2p - 1 < nkb and nkb each after that.
template <bool CAUSAL>
__device__ __forceinline__ uint32_t units_before(int p, int nkb) {
  if (!CAUSAL) return static_cast<uint32_t>(p) * static_cast<uint32_t>(nkb);
  const uint32_t c = static_cast<uint32_t>(nkb + 1) / 2u;  // pairs whose tile 0 needs 2p + 1 <= nkb blocks
  const uint32_t pp = static_cast<uint32_t>(p);
  return pp <= c ? pp * pp : c * c + (pp - c) * static_cast<uint32_t>(nkb);
}
// Pair p and block jb of unit uh of a head (inverse of units_before).
template <bool CAUSAL>
__device__ __forceinline__ void unit_pair(uint32_t uh, int nkb, int& p, int& jb) {
  const uint32_t n = static_cast<uint32_t>(nkb);
  const uint32_t c = static_cast<uint32_t>(nkb + 1) / 2u;
  if (CAUSAL && uh < c * c) {
    uint32_t r = static_cast<uint32_t>(sqrtf(static_cast<float>(uh)));  // within one of floor(sqrt(uh))
    if (r * r > uh) --r;
    if ((r + 1u) * (r + 1u) <= uh) ++r;
    p = static_cast<int>(r);
    jb = static_cast<int>(uh - r * r);
    return;
  }
  const uint32_t base = CAUSAL ? c * c : 0u;
  const uint32_t q = (uh - base) / n;
  p = static_cast<int>((CAUSAL ? c : 0u) + q);
  jb = static_cast<int>(uh - base - q * n);
}

// Share boundaries of the split schedule chosen by the host (non-causal): CTA c takes units
// [s[c], s[c+1]). s[gridDim.x] = 0 when the host gave none.
constexpr int kMaxSplitCtas = 256;
struct SplitBounds {
  uint32_t s[kMaxSplitCtas + 1];
};

// Which pieces a CTA takes. Classic: whole pairs blockIdx.x, +gridDim.x, ... (tile_info
// order). Split: a contiguous range of the U units of all heads (U < 2^31, checked by the
// host), [c U / G, (c+1) U / G) or the host's boundaries `bnd` (the same number of blocks
// each, give or take what a CTA's piece boundaries and merges cost), so no partial last wave
// is left; a pair cut by a range boundary is finished by the CTA that holds its first block,
// which processes that piece last, while the CTAs holding the rest process theirs first.
template <bool CAUSAL>
struct Schedule {
  uint32_t u, e;  // split: the remaining unit range; classic: u = next round, e = pair count
  __device__ static uint32_t start(const uint32_t* bnd, uint32_t c, uint32_t units) {
    return bnd != nullptr ? bnd[c] : static_cast<uint32_t>(static_cast<uint64_t>(c) * units / gridDim.x);
  }
  __device__ static uint32_t total_units(int BH, int num_pairs, int nkb) {
    return static_cast<uint32_t>(BH) * units_before<CAUSAL>(num_pairs, nkb);
  }
  __device__ Schedule(bool split, int BH, int num_pairs, int nkb, const uint32_t* bnd) {
    if (split) {
      const uint32_t units = total_units(BH, num_pairs, nkb);
      u = start(bnd, blockIdx.x, units);
      e = start(bnd, blockIdx.x + 1, units);
    } else {
      u = 0;
      e = static_cast<uint32_t>(BH * num_pairs);
    }
  }
  __device__ bool next(Piece& pc, bool split, int BH, int num_pairs, int nkb) {
    if (!split) {
      const int tile = classic_tile<CAUSAL>(static_cast<int>(u));
      if (tile >= static_cast<int>(e)) return false;
      const TileInfo ti = tile_info<CAUSAL>(tile, BH, num_pairs, nkb);
      pc.pair = tile;
      pc.bh = ti.bh;
      pc.q0 = ti.q0;
      pc.jb = 0;
      pc.nb0 = ti.nb0;
      pc.nb1 = ti.nb1;
      pc.kind = 0;
      ++u;
      return true;
    }
    if (u >= e) return false;
    const uint32_t hu = units_before<CAUSAL>(num_pairs, nkb);
    const uint32_t bh = u / hu;
    int p, jb;
    unit_pair<CAUSAL>(u - bh * hu, nkb, p, jb);
    const int nb0p = CAUSAL ? min(nkb, 2 * p + 1) : nkb;  // the pair's units
    const int nb1p = CAUSAL ? min(nkb, 2 * p + 2) : nkb;
    const uint32_t left = e - u;
    const int je = left < static_cast<uint32_t>(nb0p - jb) ? jb + static_cast<int>(left) : nb0p;
    pc.pair = static_cast<int>(bh) * num_pairs + p;
    pc.bh = static_cast<int>(bh);
    pc.q0 = p * 2 * kBM;
    pc.jb = jb;
    pc.nb0 = je - jb;
    pc.nb1 = pc.nb0 + (je == nb0p ? nb1p - nb0p : 0);  // tile 1's diagonal block goes with the last unit
    pc.kind = (jb == 0 && je == nb0p) ? 0 : (jb == 0 ? 1 : 2);
    u += static_cast<uint32_t>(je - jb);
    return true;
  }
};


// Share boundaries of the non-causal split schedule over G CTAs: contiguous ranges of the U
// (pair, key block) units, each pair nkb units, balanced by an estimated cost instead of the
// unit count. A range's cost, in tenths of a block: 10 per unit, 12 per further pair it
// touches (a piece boundary), 16 when it ends inside a pair whose first block it holds (it
// merges that pair's partials last), 4 when it starts inside a pair (it writes a partial).
// Weights from a per-CTA timeline at B4 H12 N2048: a block 1.3 us, a piece boundary 1.5 us, a
// merge 2 us, a partial's write about 0.5 us. The smallest target cost that a greedy fill
// (each range as long as it stays within the target) stretches over all U units.
inline void balance_split(uint32_t U, uint32_t nkb, int G, uint32_t* out) {
  auto cost = [&](uint32_t s, uint32_t e) -> uint64_t {  // range [s, e), e > s
    const uint32_t p0 = s / nkb, p1 = (e - 1u) / nkb;
    uint64_t c = 10ull * (e - s) + 12ull * (p1 - p0);
    if (e % nkb != 0u && s <= p1 * nkb) c += 16u;
    if (s % nkb != 0u) c += 4u;
    return c;
  };
  auto fill = [&](uint64_t target, uint32_t* b) {
    uint32_t s = 0;
    b[0] = 0;
    for (int c = 0; c < G; ++c) {
      uint32_t best = s;
      const uint64_t reach = target / 10u + 2u * nkb + 2u;  // no range is longer than this
      for (uint64_t e = s + 1ull; e <= U && e <= s + reach; ++e)
        if (cost(s, static_cast<uint32_t>(e)) <= target) best = static_cast<uint32_t>(e);
      b[c + 1] = best;
      s = best;
    }
    return s >= U;
  };
  uint64_t lo = 10ull * U / static_cast<uint64_t>(G), hi = 2ull * lo + 64ull;
  while (!fill(hi, out)) hi *= 2;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) / 2;
    if (fill(mid, out)) hi = mid;
    else lo = mid + 1;
  }
  fill(hi, out);
  out[G] = U;
}

// The host's share boundaries for a non-causal split launch over num_sms CTAs (all zero, so
// that the kernel divides the units evenly, for causal calls or more CTAs than the table holds),
// computed once per shape (about a millisecond) and then reused.
template <bool CAUSAL>
SplitBounds split_bounds(int BH, int M, int N, int num_sms) {
  if (CAUSAL || num_sms > kMaxSplitCtas) return SplitBounds{};
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, SplitBounds> cache;
  const int num_pairs = (M + 2 * kBM - 1) / (2 * kBM), nkb = (N + kBN - 1) / kBN;
  const auto key = std::make_tuple(BH, num_pairs, nkb, num_sms);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it == cache.end()) {
    SplitBounds b{};
    balance_split(static_cast<uint32_t>(BH) * static_cast<uint32_t>(num_pairs) * static_cast<uint32_t>(nkb),
                  static_cast<uint32_t>(nkb), num_sms, b.s);
    it = cache.emplace(key, b).first;
  }
  return it->second;
}

}  // namespace fwds
}  // namespace fa
