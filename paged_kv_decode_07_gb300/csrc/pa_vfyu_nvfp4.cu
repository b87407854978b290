// pa_vfyu_nvfp4.cu -- instantiations of the tcgen05 verify kernel for the
// NVFP4 KV format.
#include "pa_verify_umma.cuh"

namespace pa {
cudaError_t launch_verify_umma_nvfp4(const AttnParams &p, int max_items, cudaStream_t s) {
  return umma::launch_dtype<PA_KV_NVFP4>(p, max_items, s);
}
}  // namespace pa
