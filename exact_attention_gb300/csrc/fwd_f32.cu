#include "fa_internal.cuh"
namespace fa {
cudaError_t launch_fwd_f32(const void*, const void*, const void*, void*, float*, int, int, int, int, float, bool,
                           const LaunchCtx&) { return cudaErrorNotSupported; }
}
