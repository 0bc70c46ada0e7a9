#include "fa_internal.cuh"
namespace fa {
cudaError_t launch_bwd(const void*, const void*, const void*, const void*, const void*, const float*, void*, void*,
                       void*, float*, int, int, int, int, float, bool, int, const LaunchCtx&) {
  return cudaErrorNotSupported;
}
}
