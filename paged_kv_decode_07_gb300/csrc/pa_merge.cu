// pa_merge.cu -- log-sum-exp merge of split-K partials ("split-KV merge",
// "vLLM Fork with focus on GB10 Homelabs", "Acknowledgments").
//
// For one output row with partials (o_p, lse_p), lse natural-log and -inf
// for an empty partial:  M = max lse_p,  w_p = exp(lse_p - M),
// out = sum w_p o_p / sum w_p,  lse = M + ln sum w_p.  One CTA per row;
// threads split the head dim in float4 chunks, so each partial row is read
// once, coalesced.
#include "pa_internal.cuh"

namespace pa {
namespace {



__device__ __forceinline__ void store4(void *out, int out_fp32, size_t off, float4 v) {
  if (out_fp32) {
    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + off) = v;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + off) = u;
  }
}

// Merges `parts` partials of one row with one CTA of kThreads threads.
// po points at partial 0 of the row, consecutive partials `pstride` floats
// apart; pl likewise with lstride.  The lse values are read once (kept in
// shared memory for the first kChunk partials) and the weights
// exp(lse_p - M) computed once per partial into shared memory (chunks of
// kChunk).  The threads form kThreads / (D / 4) groups, each thread owning
// one float4 column: group k accumulates partials k, k + groups, ... (eight
// loads in flight per step), so a row with hundreds of partials (a 262K-key
// sequence split into partitions) is read by the whole CTA at once; the
// groups' sums are then added in fixed order.
constexpr int kThreads = 256;
constexpr int kChunk = 512;

__device__ void merge_row(const float *po, size_t pstride, const float *pl, size_t lstride,
                          int parts, int D, void *out, int out_fp32, size_t out_off,
                          float *lse_out, size_t lse_off) {
  __shared__ float s_w[kChunk];
  __shared__ float s_l[kChunk];   // lse of the first kChunk partials
  __shared__ float s_red[kThreads / 32];
  __shared__ float s_M;
  __shared__ float4 s_acc[kThreads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float M = kNegInf;
  for (int q = tid; q < parts; q += kThreads) {
    const float l = pl[(size_t)q * lstride];
    if (q < kChunk) s_l[q] = l;
    M = fmaxf(M, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  if (tid == 0) {
    float m = s_red[0];
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, s_red[w]);
    s_M = m;
  }
  __syncthreads();
  M = s_M;
  if (M == kNegInf) {
    for (int d = tid * 4; d < D; d += kThreads * 4)
      store4(out, out_fp32, out_off + d, make_float4(0, 0, 0, 0));
    if (lse_out && tid == 0) lse_out[lse_off] = kNegInf;
    return;
  }
  const int cols = D / 4;                       // float4 columns (D <= 1024: cols <= kThreads)
  const int groups = max(1, kThreads / cols);   // partial groups
  const int col = tid % cols, grp = tid / cols;
  const bool active = grp < groups && col < cols;
  float4 acc = make_float4(0, 0, 0, 0);
  float wsum = 0.f;
  for (int q0 = 0; q0 < parts; q0 += kChunk) {
    const int n = min(kChunk, parts - q0);
    __syncthreads();
    for (int q = tid; q < n; q += kThreads) {
      const float l = q0 == 0 ? s_l[q] : pl[(size_t)(q0 + q) * lstride];
      s_w[q] = (l == kNegInf) ? 0.f : __expf(l - M);
    }
    __syncthreads();
    if (grp == 0 || tid == 0)   // the threads that write the row or its lse
      for (int q = 0; q < n; ++q) wsum += s_w[q];
    if (!active) continue;
    const float *base = po + (size_t)q0 * pstride + 4 * col;
    int q = grp;
    for (; q + 7 * groups < n; q += 8 * groups) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = *reinterpret_cast<const float4 *>(base + (size_t)(q + u * groups) * pstride);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float w = s_w[q + u * groups];
        if (w != 0.f) {   // an empty partial may hold anything
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
        }
      }
    }
    for (; q < n; q += groups) {
      const float w = s_w[q];
      if (w == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4 *>(base + (size_t)q * pstride);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
  // the groups' sums of each column, added in group order
  s_acc[tid] = acc;
  __syncthreads();
  if (grp == 0 && col < cols) {
    float4 t = s_acc[col];
    for (int k = 1; k < groups; ++k) {
      const float4 u = s_acc[k * cols + col];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float inv = 1.f / wsum;
    store4(out, out_fp32, out_off + 4 * col, make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv));
  }
  if (lse_out && tid == 0) lse_out[lse_off] = M + __logf(wsum);
}

// rows of a planned call: (b, i, hq), one CTA each
__global__ void __launch_bounds__(kThreads) merge_plan_kernel(const AttnParams p) {
  griddep_wait();   // the attention kernel's outputs and partials are complete
  const int row = blockIdx.x;
  const int hq = row % p.Hq;
  const int bi = row / p.Hq;
  const int i = bi % p.Q, b = bi / p.Q;
  const int g = hq % p.G, kvh = hq / p.G;
  int u, r;
  if (p.virt == 1) {
    u = b * p.Q + i;
    r = g;
  } else if (p.virt == 2) {
    const int gr = i * p.G + g;   // row of the sequence's q_len * G
    u = b * p.RG + gr / p.R;
    r = gr % p.R;
  } else {
    u = b;
    r = i * p.G + g;
  }
  const UnitInfo ui = p.units[u];
  const int D = p.kv.D;
  if (ui.parts == 1) return;   // written by the attention kernel
  // parts == 0: nothing to attend.  A plan that did not fit the workspace
  // (flagged by the planner; no item ran) must not read past the slots.
  if (ui.parts == 0 || ui.slot_base < 0 || ui.slot_base + ui.parts > p.max_slots) {
    for (int d = threadIdx.x * 4; d < D; d += kThreads * 4)
      store4(p.out, p.out_fp32, (size_t)row * D + d, make_float4(0, 0, 0, 0));
    if (p.lse_out && threadIdx.x == 0) p.lse_out[row] = kNegInf;
    return;
  }
  const size_t slot_rows = (size_t)p.kv.hkv * p.R;
  const size_t prow = ((size_t)ui.slot_base * p.kv.hkv + kvh) * p.R + r;
  merge_row(p.part_o + prow * D, slot_rows * D, p.part_lse + prow, slot_rows, ui.parts, D, p.out,
            p.out_fp32, (size_t)row * D, p.lse_out, row);
}

// public pa_merge: part_out [S, R, D], part_lse [S, R]
__global__ void __launch_bounds__(kThreads)
    merge_dense_kernel(const float *po, const float *pl, int S, int R, int D, void *out,
                       int out_fp32, float *lse_out) {
  const int row = blockIdx.x;
  merge_row(po + (size_t)row * D, (size_t)R * D, pl + row, (size_t)R, S, D, out, out_fp32,
            (size_t)row * D, lse_out, row);
}

}  // namespace

cudaError_t launch_merge_plan(const AttnParams &p, cudaStream_t s) {
  const long long rows = (long long)p.B * p.Q * p.Hq;
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_pdl(merge_plan_kernel, (unsigned)rows, kThreads, 0, s, p);
}

cudaError_t launch_merge_dense(const float *po, const float *pl, int S, int R, int D, void *out,
                               int out_fp32, float *lse_out, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  merge_dense_kernel<<<R, kThreads, 0, s>>>(po, pl, S, R, D, out, out_fp32, lse_out);
  return cudaGetLastError();
}

}  // namespace pa
