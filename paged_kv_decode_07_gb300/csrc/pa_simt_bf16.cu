// pa_simt_bf16.cu -- instantiations of the CUDA-core decode kernel for the
// bf16 KV format (one translation unit per format so they compile in
// parallel).
#include "pa_decode_simt.cuh"

namespace pa {
cudaError_t launch_decode_simt_bf16(const AttnParams &p, int grid, cudaStream_t s) {
  return simt::launch_dtype<PA_KV_BF16>(p, grid, s);
}
}  // namespace pa
