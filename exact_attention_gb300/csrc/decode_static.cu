// fa_decode_static: decode whose split scratch the library owns.
//
// Some callers cannot allocate device memory at the moment they decode: code
// that runs under a caching or arena allocator that must not grow, a runtime
// that accounts for every buffer itself, or a C caller that has no allocator
// of its own at that point. fa_decode_static serves them: the split partials
// live in g_decode_scratch, a fixed array in the library's device image that
// every GPU using it holds until the process exits.
//
// The array has this translation unit to itself, so with lazy module loading
// (the CUDA default) a device maps it only once fa_decode_static runs there,
// not when a process uses the library's other entry points.
#include <cstdio>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kMaxScratchDevices = 64;
constexpr size_t kStaticScratchFloats = static_cast<size_t>(4) << 20;  // 16 MiB of float32

static __device__ __align__(256) float g_decode_scratch[kStaticScratchFloats];

std::mutex g_scratch_mutex;
float* g_scratch_ptr[kMaxScratchDevices] = {};

// Once per device, with that device current: the device address of the array.
// In host code the array's name only stands for it; the kernels must be given
// this address instead.
fa_status static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail_msg(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxScratchDevices) return fail_msg(FA_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return cuda_fail_msg(e, "cudaGetSymbolAddress(decode scratch)");
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_decode_static(const void* q, const void* Kcache, const void* Vcache, void* O, int B, int H,
                                      int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream) {
  if (B > 0 && H > 0 && D > 0 && n_splits > 0) {
    const size_t need = static_cast<size_t>(B) * H * n_splits * (D + 2);
    if (need > fa::kStaticScratchFloats) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "fa_decode_static: B*H*n_splits*(D+2) = %zu floats exceeds the library's fixed scratch of %zu "
               "floats (16 MiB); use fewer splits or fa_decode with a caller workspace",
               need, fa::kStaticScratchFloats);
      return fa::fail_msg(FA_ERR_INVALID, msg);
    }
  }
  float* ws = nullptr;
  if (B > 0 && H > 0) {
    const fa_status s = fa::static_scratch(&ws);
    if (s != FA_OK) return s;
  }
  // the rest of the checks and the launch are fa_decode's
  return fa::decode_entry(q, Kcache, Vcache, O, nullptr, ws, B, H, 1, N, D, scale, n_splits, dtype, stream,
                          "fa_decode_static");
}
