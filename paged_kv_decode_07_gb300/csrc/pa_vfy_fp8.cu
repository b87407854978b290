// pa_vfy_fp8.cu -- instantiations of the dense-tile verify kernel for the
// FP8-E4M3 KV format.
#include "pa_verify_mma.cuh"

namespace pa {
cudaError_t launch_verify_fp8(const AttnParams &p, int grid, cudaStream_t s) {
  return vfy::launch_dtype<PA_KV_FP8>(p, grid, s);
}
}  // namespace pa
