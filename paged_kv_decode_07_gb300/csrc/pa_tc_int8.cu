// pa_tc_int8.cu -- instantiations of the tensor-core decode kernel for the
// int8 KV format (one translation unit per format so they compile in
// parallel).
#include "pa_decode_mma.cuh"

namespace pa {
cudaError_t launch_decode_tc_int8(const AttnParams &p, int grid, cudaStream_t s) {
  return tc::launch_dtype<PA_KV_INT8>(p, grid, s);
}
cudaError_t launch_decode_tc_cluster_int8(const AttnParams &p, int P, cudaStream_t s) {
  return tc::launch_cluster_dtype<PA_KV_INT8>(p, P, s);
}
int decode_tc_occupancy_int8(int D, int R) { return tc::occupancy_dtype<PA_KV_INT8>(D, R); }
}  // namespace pa
