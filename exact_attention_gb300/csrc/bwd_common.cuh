// Definitions shared by the backward kernels' translation units (bwd.cu: delta, dK/dV, dQ, the
// fused pass; bwd_pair.cu: the CTA-pair dK/dV and dQ kernels).
#pragma once
#include <cstdint>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kT = 128;          // tile rows (keys or queries) and streamed block rows
constexpr int kChunkB = 16384;   // 128 rows x 128 bytes, one swizzled chunk
constexpr float kLog2eB = 1.4426950408889634f;

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

}  // namespace
}  // namespace fa
