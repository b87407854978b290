// pa_merge.cu -- log-sum-exp merge of split-K partials ("split-KV merge",
// "vLLM Fork with focus on GB10 Homelabs", "Acknowledgments").
//
// For one output row with partials (o_p, lse_p), lse natural-log and -inf
// for an empty partial:  M = max lse_p,  w_p = exp(lse_p - M),
// out = sum w_p o_p / sum w_p,  lse = M + ln sum w_p.  One warp per row;
// lanes split the head dim in float4 chunks, so each partial row is read
// once, coalesced.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kWarpsPerCta = 8;


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

// Merges `parts` partials of one row.  po points at partial 0 of the row,
// consecutive partials `pstride` floats apart; pl likewise with lstride.
__device__ void merge_row(const float *po, size_t pstride, const float *pl, size_t lstride,
                          int parts, int D, void *out, int out_fp32, size_t out_off,
                          float *lse_out, size_t lse_off) {
  const int lane = threadIdx.x & 31;
  float M = kNegInf;
  for (int q = lane; q < parts; q += 32) M = fmaxf(M, pl[(size_t)q * lstride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M == kNegInf) {
    for (int d = lane * 4; d < D; d += 128) store4(out, out_fp32, out_off + d, make_float4(0, 0, 0, 0));
    if (lse_out && lane == 0) lse_out[lse_off] = kNegInf;
    return;
  }
  float wsum = 0.f;
  for (int d0 = 0; d0 < D; d0 += 128) {
    const int d = d0 + lane * 4;
    float4 acc = make_float4(0, 0, 0, 0);
    float ws = 0.f;
    for (int q = 0; q < parts; ++q) {
      const float l = pl[(size_t)q * lstride];
      if (l == kNegInf) continue;
      const float w = __expf(l - M);
      ws += w;
      if (d < D) {
        float4 v = *reinterpret_cast<const float4 *>(po + (size_t)q * pstride + d);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
    wsum = ws;
    if (d < D) {
      const float inv = 1.f / ws;
      store4(out, out_fp32, out_off + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
  }
  if (lse_out && lane == 0) lse_out[lse_off] = M + __logf(wsum);
}

// rows of a planned call: (b, i, hq)
__global__ void __launch_bounds__(kWarpsPerCta * 32) merge_plan_kernel(const AttnParams p) {
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int rows = p.B * p.Q * p.Hq;
  if (row >= rows) return;
  const int hq = row % p.Hq;
  const int bi = row / p.Hq;
  const int i = bi % p.Q, b = bi / p.Q;
  const int g = hq % p.G, kvh = hq / p.G;
  const int u = p.virt ? b * p.Q + i : b;
  const int r = p.virt ? g : i * p.G + g;
  const UnitInfo ui = p.units[u];
  const int D = p.kv.D;
  if (ui.parts == 1) return;   // written by the attention kernel
  // parts == 0: nothing to attend.  A plan that did not fit the workspace
  // (flagged by the planner; no item ran) must not read past the slots.
  if (ui.parts == 0 || ui.slot_base < 0 || ui.slot_base + ui.parts > p.max_slots) {
    const int lane = threadIdx.x & 31;
    for (int d = lane * 4; d < D; d += 128)
      store4(p.out, p.out_fp32, (size_t)row * D + d, make_float4(0, 0, 0, 0));
    if (p.lse_out && lane == 0) p.lse_out[row] = kNegInf;
    return;
  }
  const size_t slot_rows = (size_t)p.kv.hkv * p.R;
  const size_t prow = ((size_t)ui.slot_base * p.kv.hkv + kvh) * p.R + r;
  merge_row(p.part_o + prow * D, slot_rows * D, p.part_lse + prow, slot_rows, ui.parts, D, p.out,
            p.out_fp32, (size_t)row * D, p.lse_out, row);
}

// public pa_merge: part_out [S, R, D], part_lse [S, R]
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    merge_dense_kernel(const float *po, const float *pl, int S, int R, int D, void *out,
                       int out_fp32, float *lse_out) {
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (row >= R) return;
  merge_row(po + (size_t)row * D, (size_t)R * D, pl + row, (size_t)R, S, D, out, out_fp32,
            (size_t)row * D, lse_out, row);
}

}  // namespace

cudaError_t launch_merge_plan(const AttnParams &p, cudaStream_t s) {
  const int rows = p.B * p.Q * p.Hq;
  if (rows == 0) return cudaSuccess;
  merge_plan_kernel<<<(rows + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge_dense(const float *po, const float *pl, int S, int R, int D, void *out,
                               int out_fp32, float *lse_out, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  merge_dense_kernel<<<(R + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(
      po, pl, S, R, D, out, out_fp32, lse_out);
  return cudaGetLastError();
}

}  // namespace pa
