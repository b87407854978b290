// pa_vfy_nvfp4.cu -- instantiations of the dense-tile verify kernel for the
// nvfp4 KV format.
#include "pa_verify_mma.cuh"

namespace pa {
cudaError_t launch_verify_nvfp4(const AttnParams &p, int grid, cudaStream_t s) {
  return vfy::launch_dtype<PA_KV_NVFP4>(p, grid, s);
}
}  // namespace pa
