// pa_tc_nvfp4.cu -- instantiations of the tensor-core decode kernel for the
// nvfp4 KV format (one translation unit per format so they compile in
// parallel).
#include "pa_decode_mma.cuh"

namespace pa {
cudaError_t launch_decode_tc_nvfp4(const AttnParams &p, int grid, cudaStream_t s) {
  return tc::launch_dtype<PA_KV_NVFP4>(p, grid, s);
}
cudaError_t launch_decode_tc_cluster_nvfp4(const AttnParams &p, int P, cudaStream_t s) {
  return tc::launch_cluster_dtype<PA_KV_NVFP4>(p, P, s);
}
int decode_tc_occupancy_nvfp4(int D, int R) { return tc::occupancy_dtype<PA_KV_NVFP4>(D, R); }
}  // namespace pa
