// Quantisation of the FP8 forward's operands ("Flash Attention" notes, section
// "FlashAttention 3", the FP8 bullets): incoherent processing of Q and K with the
// Hadamard-times-sign matrix M = diag(signs) H / 8 (d = 64), then E4M3 with one scale per
// 128-row block; V with one scale per (batch, head), written transposed ([d][keys]) so that
// it serves as the K-major operand of P V.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kD8 = 64;
constexpr int kRowsPerBlock = 128;
constexpr float kE4M3Max = 448.f;

template <bool BF16>
__device__ __forceinline__ float half_to_f32(uint16_t h) {
  return BF16 ? __uint_as_float(static_cast<uint32_t>(h) << 16) : __half2float(__ushort_as_half(h));
}

// Largest value of v over the CTA's 128 threads (all threads get it).
__device__ __forceinline__ float block_max128(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  return v;
}

// Largest |V| of one 128-key block of one head into vmax (16-byte loads contiguous across
// each warp).
template <bool BF16>
__device__ __forceinline__ void v_block_amax(const uint16_t* __restrict__ V, float* __restrict__ vmax, int N,
                                             float* red) {
  const int nkb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
  if (static_cast<int>(blockIdx.x) >= nkb) return;  // the grid covers the longest of Q, K, V
  const size_t bh = blockIdx.y;
  const int k0 = static_cast<int>(blockIdx.x) * kRowsPerBlock;
  const int nrows = min(kRowsPerBlock, N - k0);
  const uint4* src = reinterpret_cast<const uint4*>(V + (bh * N + k0) * kD8);
  float am = 0.f;
  uint4 ld[kRowsPerBlock * kD8 / 8 / 128];
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    ld[i] = c < nrows * kD8 / 8 ? src[c] : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const uint4 v = ld[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      am = fmaxf(am, fmaxf(fabsf(half_to_f32<BF16>(static_cast<uint16_t>(w[j] & 0xFFFFu))),
                           fabsf(half_to_f32<BF16>(static_cast<uint16_t>(w[j] >> 16)))));
  }
  am = block_max128(am, red);
  if (threadIdx.x == 0) vmax[bh * nkb + blockIdx.x] = am;
}

// Q (blockIdx.z = 0) or K (1): one CTA per 128-row block of one head, one row per thread.
// x -> x diag(signs) H / 8 by a fast Walsh-Hadamard transform in registers, then the block's
// scale = amax / 448 and the E4M3 row. The block moves through shared memory in 16-byte
// pieces, so that its global loads and stores are contiguous across each warp. z = 2: V's
// per-block maxima (same launch: all three only read the inputs).
template <bool BF16>
__global__ void __launch_bounds__(128) fp8_qk_quant_kernel(const uint16_t* __restrict__ Q,
                                                           const uint16_t* __restrict__ K,
                                                           const uint16_t* __restrict__ V,
                                                           const int8_t* __restrict__ signs, uint8_t* __restrict__ Q8,
                                                           uint8_t* __restrict__ K8, float* __restrict__ sq,
                                                           float* __restrict__ sk, float* __restrict__ vmax, int M,
                                                           int N) {
  __shared__ uint32_t tile[kRowsPerBlock][kD8 / 2 + 1];  // 32 words of halves a row (+1: no bank conflicts)
  __shared__ float red[4];
  // launched as a programmatic dependent: the inputs may come from the kernel before it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();
  if (blockIdx.z == 2) {
    v_block_amax<BF16>(V, vmax, N, red);
    return;
  }
  const bool isk = blockIdx.z == 1;
  const int rows = isk ? N : M;
  const int nblk = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (static_cast<int>(blockIdx.x) >= nblk) return;  // the grid covers the longer of the two
  const size_t bh = blockIdx.y;
  const int r0 = static_cast<int>(blockIdx.x) * kRowsPerBlock;
  const int nrows = min(kRowsPerBlock, rows - r0);
  const uint4* src = reinterpret_cast<const uint4*>((isk ? K : Q) + (bh * rows + r0) * kD8);
  // eight independent 16-byte loads a thread, all in flight at once
  uint4 ld[kRowsPerBlock * kD8 / 8 / 128];
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    ld[i] = (c >> 3) < nrows ? src[c] : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    const int r = c >> 3, q = c & 7;
    const uint4 v = ld[i];
    tile[r][4 * q] = v.x;
    tile[r][4 * q + 1] = v.y;
    tile[r][4 * q + 2] = v.z;
    tile[r][4 * q + 3] = v.w;
  }
  __syncthreads();
  const int r = threadIdx.x;
  float x[kD8];
#pragma unroll
  for (int w = 0; w < kD8 / 2; ++w) {
    const uint32_t v = tile[r][w];
    x[2 * w] = half_to_f32<BF16>(static_cast<uint16_t>(v & 0xFFFFu));
    x[2 * w + 1] = half_to_f32<BF16>(static_cast<uint16_t>(v >> 16));
  }
  {  // the signs as one bit each (an int8 is negative when its top bit is set)
    const uint4* s4 = reinterpret_cast<const uint4*>(signs);
    uint32_t sw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(s4 + i);
      sw[4 * i] = v.x;
      sw[4 * i + 1] = v.y;
      sw[4 * i + 2] = v.z;
      sw[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int d = 0; d < kD8; ++d)
      x[d] = __uint_as_float(__float_as_uint(x[d]) ^ (((sw[d / 4] >> (8 * (d % 4) + 7)) & 1u) << 31));
  }
#pragma unroll
  for (int h = 1; h < kD8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < kD8; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
  float am = 0.f;
#pragma unroll
  for (int d = 0; d < kD8; ++d) {
    x[d] *= 0.125f;  // 1 / sqrt(64), exact
    am = fmaxf(am, fabsf(x[d]));
  }
  am = block_max128(am, red);  // (its barriers also order the tile's reads before the writes below)
  const float scale = am > 0.f ? am / kE4M3Max : 1.f;
  const float inv = am > 0.f ? kE4M3Max / am : 1.f;
  if (threadIdx.x == 0) (isk ? sk : sq)[bh * nblk + blockIdx.x] = scale;
  // the E4M3 row (16 words) back into the tile, then out 16 bytes at a time
#pragma unroll
  for (int p = 0; p < 16; ++p)
    tile[r][p] = ptx::pack_e4m3x2(x[4 * p] * inv, x[4 * p + 1] * inv) |
                 (ptx::pack_e4m3x2(x[4 * p + 2] * inv, x[4 * p + 3] * inv) << 16);
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>((isk ? K8 : Q8) + (bh * rows + r0) * kD8);
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 16 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    const int rr = c >> 2, q = c & 3;
    if (rr < nrows) dst[c] = make_uint4(tile[rr][4 * q], tile[rr][4 * q + 1], tile[rr][4 * q + 2], tile[rr][4 * q + 3]);
  }
}

// V of one 128-key block quantised with its head's scale and written transposed:
// Vt8[bh][d][key], rows of Npad bytes (keys past N are zero).
template <bool BF16>
__global__ void __launch_bounds__(128) fp8_v_quant_kernel(const uint16_t* __restrict__ V,
                                                          const float* __restrict__ vmax, uint8_t* __restrict__ Vt8,
                                                          float* __restrict__ sv, int N, int Npad) {
  __shared__ float tile[kRowsPerBlock][kD8 + 1];
  __shared__ float red[4];
  const int nkb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
  const size_t bh = blockIdx.y;
  const int k0 = static_cast<int>(blockIdx.x) * kRowsPerBlock;
  // launched as a programmatic dependent of the launch that wrote vmax
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::grid_dep_wait();
  float am = 0.f;
  for (int i = threadIdx.x; i < nkb; i += blockDim.x) am = fmaxf(am, vmax[bh * nkb + i]);
  am = block_max128(am, red);
  const float scale = am > 0.f ? am / kE4M3Max : 1.f;
  const float inv = am > 0.f ? kE4M3Max / am : 1.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) sv[bh] = scale;
  // the block's 128 x 64 values (contiguous in memory) into shared memory, 16 bytes per load
  const uint16_t* src = V + (bh * static_cast<size_t>(N) + k0) * kD8;
  uint4 ld[kRowsPerBlock * kD8 / 8 / 128];
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    ld[i] = k0 + c / (kD8 / 8) < N ? reinterpret_cast<const uint4*>(src)[c] : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kRowsPerBlock * kD8 / 8 / 128; ++i) {
    const int c = static_cast<int>(threadIdx.x) + 128 * i;
    const int key = c / (kD8 / 8), d0 = (c % (kD8 / 8)) * 8;
    const uint4 v = ld[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tile[key][d0 + 2 * i] = half_to_f32<BF16>(static_cast<uint16_t>(w[i] & 0xFFFFu));
      tile[key][d0 + 2 * i + 1] = half_to_f32<BF16>(static_cast<uint16_t>(w[i] >> 16));
    }
  }
  __syncthreads();
  // thread t writes column d = t / 2 for keys [64 (t % 2), 64 (t % 2) + 64) of the block
  const int d = threadIdx.x >> 1, kh = (threadIdx.x & 1) * 64;
  float x[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) x[i] = tile[kh + i][d];
  uint8_t* dst = Vt8 + (bh * kD8 + d) * static_cast<size_t>(Npad) + k0 + kh;
  uint32_t w[16];
#pragma unroll
  for (int p = 0; p < 16; ++p)
    w[p] = ptx::pack_e4m3x2(x[4 * p] * inv, x[4 * p + 1] * inv) |
           (ptx::pack_e4m3x2(x[4 * p + 2] * inv, x[4 * p + 3] * inv) << 16);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (k0 + kh + 16 * c < Npad)
      reinterpret_cast<uint4*>(dst)[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

}  // namespace

cudaError_t launch_fp8_quant(const void* Q, const void* K, const void* V, const int8_t* signs, const Fp8Ws& w, int BH,
                             int M, int N, int dtype, cudaStream_t stream) {
  const int nqb = (M + kRowsPerBlock - 1) / kRowsPerBlock, nkb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
  const auto* q = static_cast<const uint16_t*>(Q);
  const auto* k = static_cast<const uint16_t*>(K);
  const auto* v = static_cast<const uint16_t*>(V);
  // both launches are programmatic dependents of the kernel before them on the stream
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Q, K (blocks of 128 rows) and V's block maxima in one launch, then V
  cfg.gridDim = dim3(static_cast<unsigned>(nqb > nkb ? nqb : nkb), static_cast<unsigned>(BH), 3u);
  cudaError_t e = dtype == kBF16 ? cudaLaunchKernelEx(&cfg, fp8_qk_quant_kernel<true>, q, k, v, signs, w.q8, w.k8, w.sq,
                                                      w.sk, w.vmax, M, N)
                                 : cudaLaunchKernelEx(&cfg, fp8_qk_quant_kernel<false>, q, k, v, signs, w.q8, w.k8, w.sq,
                                                      w.sk, w.vmax, M, N);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(nkb), static_cast<unsigned>(BH));
  return dtype == kBF16
             ? cudaLaunchKernelEx(&cfg, fp8_v_quant_kernel<true>, v, static_cast<const float*>(w.vmax), w.vt8, w.sv, N,
                                  w.npad)
             : cudaLaunchKernelEx(&cfg, fp8_v_quant_kernel<false>, v, static_cast<const float*>(w.vmax), w.vt8, w.sv,
                                  N, w.npad);
}

}  // namespace fa
