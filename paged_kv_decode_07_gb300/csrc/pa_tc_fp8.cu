// pa_tc_fp8.cu -- instantiations of the tensor-core decode kernel for the
// FP8-E4M3 KV format (one translation unit per format so they compile in
// parallel).
#include "pa_decode_mma.cuh"

namespace pa {
cudaError_t launch_decode_tc_fp8(const AttnParams &p, int grid, cudaStream_t s) {
  return tc::launch_dtype<PA_KV_FP8>(p, grid, s);
}
cudaError_t launch_decode_tc_cluster_fp8(const AttnParams &p, int P, cudaStream_t s) {
  return tc::launch_cluster_dtype<PA_KV_FP8>(p, P, s);
}
int decode_tc_occupancy_fp8(int D, int R) { return tc::occupancy_dtype<PA_KV_FP8>(D, R); }
}  // namespace pa
