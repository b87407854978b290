// pa_vfyu_fp8.cu -- instantiations of the tcgen05 verify kernel for the
// FP8-E4M3 KV format.
#include "pa_verify_umma.cuh"

namespace pa {
cudaError_t launch_verify_umma_fp8(const AttnParams &p, int max_items, cudaStream_t s) {
  return umma::launch_dtype<PA_KV_FP8>(p, max_items, s);
}
}  // namespace pa
