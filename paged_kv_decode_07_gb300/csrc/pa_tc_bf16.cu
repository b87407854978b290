// pa_tc_bf16.cu -- instantiations of the tensor-core decode kernel for the
// bf16 KV format (ldmatrix fragments, no dequantisation).
#include "pa_decode_mma.cuh"

namespace pa {
cudaError_t launch_decode_tc_bf16(const AttnParams &p, int grid, cudaStream_t s) {
  return tc::launch_dtype<PA_KV_BF16>(p, grid, s);
}
cudaError_t launch_decode_tc_cluster_bf16(const AttnParams &p, int P, cudaStream_t s) {
  return tc::launch_cluster_dtype<PA_KV_BF16>(p, P, s);
}
int decode_tc_occupancy_bf16(int D, int R) { return tc::occupancy_dtype<PA_KV_BF16>(D, R); }
}  // namespace pa
