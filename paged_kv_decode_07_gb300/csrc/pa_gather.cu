// pa_gather.cu -- debug kernel: gather through the block table and
// dequantise to fp32 exactly as the attention kernels' register dequant
// does (same helpers), so that block-table indexing and the formats can be
// checked bit for bit.
//   bf16  : widened exactly.
//   int8  : (float)code * (float)scale_fp16                  (exact product)
//   NVFP4 : ((e2m1 * e4m3) computed in f16, exact) * global (one fp32 round)
//   FP8   : e4m3 (exact in f16) * global                     (one fp32 round)
// PagedAttention addressing (Kwon et al., cited on "vLLM Fork with focus on
// GB10 Homelabs", "About"): token t of sequence b is slot t % 16 of block
// block_tables[b][t / 16].
#include "pa_internal.cuh"

namespace pa {
namespace {

// one warp per (b, kvh, t); lanes over D in chunks of 8
__global__ void gather_kernel(KvView kv, const int *tables, int stride, const int *seq_lens, int B,
                              int max_len, float *k_out, float *v_out, uint32_t *hdr) {
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long total = (long long)B * kv.hkv * max_len;
  if (w >= total) return;
  const int t = (int)(w % max_len);
  const int h = (int)((w / max_len) % kv.hkv);
  const int b = (int)(w / ((long long)max_len * kv.hkv));
  const int D = kv.D;
  float *ko = k_out + (size_t)w * D, *vo = v_out + (size_t)w * D;
  int L = seq_lens[b];
  if (L > stride * kBlock) L = stride * kBlock;
  int phys = -1;
  if (t < L) {
    phys = tables[(size_t)b * stride + t / kBlock];
    if (phys < 0 || phys >= kv.num_blocks) {
      if (lane == 0) set_err(hdr, PA_ERRF_BAD_BLOCK_ID);
      phys = -1;
    }
  }
  for (int d0 = lane * 8; d0 < D; d0 += 256) {
    float kf[8], vf[8];
    if (phys < 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) kf[j] = vf[j] = 0.f;
    } else {
      const size_t row = ((size_t)phys * kv.hkv + h) * kBlock + (t % kBlock);
      for (int which = 0; which < 2; ++which) {
        float *f = which ? vf : kf;
        const void *data = which ? kv.v : kv.k;
        const void *sc = which ? kv.vs : kv.ks;
        if (kv.dtype == PA_KV_BF16) {
          uint4 u = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(data) +
                                                     row * D + d0);
          uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 x = bf16x2_to_f2(w4[j]);
            f[2 * j] = x.x;
            f[2 * j + 1] = x.y;
          }
        } else if (kv.dtype == PA_KV_INT8) {
          uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const int8_t *>(data) + row * D + d0);
          s8x4_to_f4(u.x, f);
          s8x4_to_f4(u.y, f + 4);
          const float s = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sc)[row]);
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = f[j] * s;
        } else if (kv.dtype == PA_KV_FP8) {
          uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(data) +
                                                     row * D + d0);
          const float g = which ? kv.vg : kv.kg;
          uint32_t w2[2] = {u.x, u.y};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 x = h2u_to_f2(e4m3x2_u16_to_h2(w2[j >> 1] >> (16 * (j & 1))));
            f[2 * j] = x.x * g;
            f[2 * j + 1] = x.y * g;
          }
        } else {
          uint32_t u = *reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint8_t *>(data) +
                                                           row * (D / 2) + d0 / 2);
          uint32_t s2 = e4m3_to_h2_dup(reinterpret_cast<const uint8_t *>(sc)[row * (D / 16) + d0 / 16]);
          const float g = which ? kv.vg : kv.kg;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 x = h2u_to_f2(hmul2_u32(e2m1x2_to_h2((u >> (8 * j)) & 0xffu), s2));
            f[2 * j] = x.x * g;
            f[2 * j + 1] = x.y * g;
          }
        }
      }
    }
    *reinterpret_cast<float4 *>(ko + d0) = make_float4(kf[0], kf[1], kf[2], kf[3]);
    *reinterpret_cast<float4 *>(ko + d0 + 4) = make_float4(kf[4], kf[5], kf[6], kf[7]);
    *reinterpret_cast<float4 *>(vo + d0) = make_float4(vf[0], vf[1], vf[2], vf[3]);
    *reinterpret_cast<float4 *>(vo + d0 + 4) = make_float4(vf[4], vf[5], vf[6], vf[7]);
  }
}

}  // namespace

cudaError_t launch_gather(const KvView &kv, const int *tables, int stride, const int *seq_lens,
                          int B, int max_len, float *k_out, float *v_out, uint32_t *hdr,
                          cudaStream_t s) {
  const long long warps = (long long)B * kv.hkv * max_len;
  if (warps == 0) return cudaSuccess;
  const int wpc = 8;
  const long long grid = (warps + wpc - 1) / wpc;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  gather_kernel<<<(unsigned)grid, wpc * 32, 0, s>>>(kv, tables, stride, seq_lens, B, max_len, k_out,
                                                    v_out, hdr);
  return cudaGetLastError();
}

}  // namespace pa
