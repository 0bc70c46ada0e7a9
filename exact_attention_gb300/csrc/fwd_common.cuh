// Pieces shared by the half-precision forward kernels: the tile order over
// (batch, head, query-tile pair) and packed f32 arithmetic for the softmax.
#pragma once
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace fwdc {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per block

struct TileInfo {
  int bh, q0, nb0, nb1;
};

template <bool CAUSAL>
__device__ __forceinline__ TileInfo tile_info(int tile, int BH, int num_pairs, int nkb) {
  TileInfo ti;
  int pair;
  if (CAUSAL) {  // heads fastest, heaviest (last) pairs first
    const int pr = tile / BH;
    ti.bh = tile - pr * BH;
    pair = num_pairs - 1 - pr;
  } else {       // pairs of one head adjacent
    ti.bh = tile / num_pairs;
    pair = tile - ti.bh * num_pairs;
  }
  ti.q0 = pair * 2 * kBM;
  if (CAUSAL) {
    ti.nb0 = min(nkb, ti.q0 / kBN + 1);
    ti.nb1 = min(nkb, (ti.q0 + kBM) / kBN + 1);
  } else {
    ti.nb0 = nkb;
    ti.nb1 = nkb;
  }
  return ti;
}

// The CTA's r-th pair of the classic schedule (whole pairs, one CTA per SM): round-robin
// over the tile_info order, every other round reversed when causal (serpentine), so the CTA
// that took one of the heaviest pairs of a round takes one of the lightest of the next.
template <bool CAUSAL>
__device__ __forceinline__ int classic_tile(int r) {
  const int c = (CAUSAL && (r & 1)) ? static_cast<int>(gridDim.x - 1u - blockIdx.x) : static_cast<int>(blockIdx.x);
  return r * static_cast<int>(gridDim.x) + c;
}

// packed f32 arithmetic lives in ptx.cuh
using ptx::fadd2;
using ptx::ffma2;
using ptx::fmax3;

// Scores of keys past N, or past the query when causal, become -inf.
template <bool CAUSAL>
__device__ __forceinline__ void mask32(uint32_t* r, int key0, int N, int row) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int key = key0 + i;
    if (key >= N || (CAUSAL && key > row)) r[i] = __float_as_uint(-INFINITY);
  }
}

}  // namespace fwdc
}  // namespace fa
