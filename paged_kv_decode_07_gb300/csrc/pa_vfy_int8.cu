// pa_vfy_int8.cu -- instantiations of the dense-tile verify kernel for the
// int8 KV format.
#include "pa_verify_mma.cuh"

namespace pa {
cudaError_t launch_verify_int8(const AttnParams &p, int grid, cudaStream_t s) {
  return vfy::launch_dtype<PA_KV_INT8>(p, grid, s);
}
}  // namespace pa
