// pa_launch.h -- host-side entry points of the kernels, one per translation
// unit, called by the C ABI in pa_api.cu (kept apart from the device
// helpers of pa_internal.cuh so that adding a kernel does not touch the
// headers the existing kernels are built from).
#pragma once

#include "pa_internal.cuh"

namespace pa {

cudaError_t launch_plan(const PlanParams &pp, cudaStream_t s);
cudaError_t launch_decode_simt(const AttnParams &p, int grid, cudaStream_t s);
int simt_supported(int dtype, int D, int R);
cudaError_t launch_merge_plan(const AttnParams &p, cudaStream_t s);
cudaError_t launch_merge_dense(const float *po, const float *pl, int S, int R, int D, void *out,
                               int out_fp32, float *lse_out, cudaStream_t s);
cudaError_t launch_means(const KvView &kv, const int *tables, int stride, const int *seq_lens,
                         const int *first, int count, int B, int sb, int max_nsb, float *means,
                         uint32_t *hdr, cudaStream_t s);
cudaError_t launch_sparse_select(const KvView &kv, const __nv_bfloat16 *q, int Hq,
                                 const int *tables, int stride, const int *seq_lens, int B, int sb,
                                 int max_nsb, int top_k, const float *means, float *scores,
                                 int *selected, int *vtables, int vstride, int *vlens,
                                 uint32_t *err, cudaStream_t s);
int wo_splits(int M, int K, int N, int requested);
cudaError_t launch_wo(const float *o, int M, int K, const void *w, int N, int splits, float *part,
                      void *y, int y_fp32, uint32_t *hdr, cudaStream_t s);
cudaError_t launch_append(const KvView &kv, const void *k_new, const void *v_new, int T,
                          const int64_t *slots, uint32_t *hdr, cudaStream_t s);
cudaError_t launch_gather(const KvView &kv, const int *tables, int stride, const int *seq_lens,
                          int B, int max_len, float *k_out, float *v_out, uint32_t *hdr,
                          cudaStream_t s);

}  // namespace pa
