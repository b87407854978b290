// pa_decode_simt.cuh -- split-K paged decode attention on the CUDA cores.
//
// One CTA (4 warps) takes one work item = (unit, kv head, range of 16-token
// blocks).  Each warp streams its share of the item's tokens through a
// private ring of shared-memory stages filled by 1-D bulk copies (TMA
// engine): a (block, kv head) tile is contiguous in the [NB, Hkv, 16, D]
// pool, so 8 tokens x D of K, the same of V and their scales are four
// copies.  PagedAttention's gather (Kwon et al., cited on "vLLM Fork with
// focus on GB10 Homelabs", "About") is the table lookup that picks the
// source address; the "TMA plane loading" and inline KV dequant of the b12x
// kernel ("Acknowledgments", same page) are the prior art this follows.
//
// Scores (the QK^T contraction) per warp iteration of 8 tokens per row
// group: lane (rg, dl) owns head-dim slice [8 dl, 8 dl + 8) and keeps the
// G query heads of that slice in registers (pre-scaled by softmax_scale *
// log2 e).  It computes partial dot products for 8 tokens x G heads, then a
// shuffle reduce-scatter sums them across the lanes that share a row: three
// halving steps over tokens (lanes read the tokens in an order XOR-permuted
// by their lane bits, so each step sends registers [n/2, n) and keeps
// [0, n/2) with no selects) and one or two steps over heads.  Afterwards
// each lane holds complete scores for one token and G / 2 (or G / 4) heads.
//
// Online softmax (flash-decoding) runs in the log2 domain with a lazy
// rescale: the running max only moves when a new score exceeds it by more
// than 8 (p <= 256 stays exact in fp32), so the accumulator rescale is a
// rare event.  PV: probabilities go through shared memory as broadcasts;
// each lane accumulates o[G][8] for its slice in fp32 with packed f32x2
// FMAs.  At the end the 4 warps' (m, l, o) are merged in shared memory and
// the item writes either the final output (single-partition sequences) or
// a normalised partial plus its LSE for the merge kernel.
//
// Dequant in registers: bf16 widened exactly; int8 codes widened exactly
// (magic-number byte permute), the per-token fp16 scale multiplies the
// score (K) or the probability (V); NVFP4 codes via cvt e2m1x2 -> f16x2 and
// one f16x2 multiply by the E4M3 block scale (exact), the per-tensor global
// scale folded into the query (K) and the output (V).
#pragma once

#include "pa_internal.cuh"

namespace pa {
namespace simt {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

template <int DT, int D>
struct Geo {
  static constexpr int LPR = D / 8;            // lanes per token row
  static constexpr int RG = 32 / LPR;          // row groups per warp
  static constexpr int TB = (D == 256) ? 2 : 1;  // log2(LPR) - 3
  static constexpr int TOK = 8 * RG;           // tokens per warp iteration (one stage)
  static constexpr int IPB = kBlock / TOK;     // iterations per 16-token block
  static constexpr int ROW_BYTES =
      DT == PA_KV_BF16 ? 2 * D : ((DT == PA_KV_INT8 || DT == PA_KV_FP8) ? D : D / 2);
  static constexpr int CODE_BYTES = TOK * ROW_BYTES;
  static constexpr int SROW_BYTES = DT == PA_KV_INT8 ? 2 : (DT == PA_KV_NVFP4 ? D / 16 : 0);
  static constexpr int SCALE_BYTES = TOK * SROW_BYTES;
  static constexpr int STAGE = 2 * (CODE_BYTES + SCALE_BYTES);
  static constexpr int NSTAGE = DT == PA_KV_NVFP4 ? 6 : 3;
  static constexpr int WARP_BYTES = NSTAGE * STAGE;
  static constexpr int SMEM = kWarps * WARP_BYTES;
  static_assert(CODE_BYTES % 16 == 0 && SCALE_BYTES % 16 == 0, "bulk copy granularity");
};

// 8 consecutive head-dim values of token row t of a stage, as 4 float2.
// int8: raw codes (scale applied by the caller); NVFP4: e2m1 * block scale;
// FP8: e4m3 values (the per-tensor scale is folded into q and the output).
template <int DT, int D>
__device__ __forceinline__ void load8(const uint8_t *codes, const uint8_t *scales, int t, int dl,
                                      float2 (&f)[4]) {
  using G_ = Geo<DT, D>;
  if constexpr (DT == PA_KV_BF16) {
    uint4 u = *reinterpret_cast<const uint4 *>(codes + t * G_::ROW_BYTES + dl * 16);
    f[0] = bf16x2_to_f2(u.x);
    f[1] = bf16x2_to_f2(u.y);
    f[2] = bf16x2_to_f2(u.z);
    f[3] = bf16x2_to_f2(u.w);
  } else if constexpr (DT == PA_KV_FP8) {
    uint2 u = *reinterpret_cast<const uint2 *>(codes + t * G_::ROW_BYTES + dl * 8);
    f[0] = h2u_to_f2(e4m3x2_u16_to_h2(u.x));
    f[1] = h2u_to_f2(e4m3x2_u16_to_h2(u.x >> 16));
    f[2] = h2u_to_f2(e4m3x2_u16_to_h2(u.y));
    f[3] = h2u_to_f2(e4m3x2_u16_to_h2(u.y >> 16));
  } else if constexpr (DT == PA_KV_INT8) {
    uint2 u = *reinterpret_cast<const uint2 *>(codes + t * G_::ROW_BYTES + dl * 8);
    float x[8];
    s8x4_to_f4(u.x, x);
    s8x4_to_f4(u.y, x + 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = make_float2(x[2 * j], x[2 * j + 1]);
  } else {
    uint32_t u = *reinterpret_cast<const uint32_t *>(codes + t * G_::ROW_BYTES + dl * 4);
    uint32_t s = scales[t * G_::SROW_BYTES + (dl >> 1)];
    uint32_t s2 = e4m3_to_h2_dup(s);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = h2u_to_f2(hmul2_u32(e2m1x2_to_h2((u >> (8 * j)) & 0xffu), s2));
  }
}

template <int DT, int D, int R>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const AttnParams p) {
  using Gm = Geo<DT, D>;
  constexpr int LPR = Gm::LPR, RG = Gm::RG, TB = Gm::TB, TOK = Gm::TOK, IPB = Gm::IPB;
  constexpr int NSTAGE = Gm::NSTAGE;
  // head split schedule after the token steps
  constexpr bool SPLIT1 = (TB >= 1) && (R % 2 == 0);
  constexpr int N1 = SPLIT1 ? R / 2 : R;
  constexpr bool SPLIT2 = (TB >= 2) && (N1 % 2 == 0);
  constexpr int NH = (TB >= 2) ? (SPLIT2 ? N1 / 2 : N1) : N1;   // heads held per lane
  constexpr float kRescale = 8.0f;


  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][NSTAGE];
  __shared__ __align__(16) float pbuf[kWarps][TOK][8];
  __shared__ __align__(16) float red[kWarps][8];
  __shared__ float s_m[kWarps][8], s_l[kWarps][8];

  griddep_launch();   // the merge may start launching once every CTA has begun
  griddep_wait();     // the plan of this call is complete
  const uint32_t num_items = p.hdr[HDR_NUM_ITEMS];
  if (blockIdx.x >= num_items) return;
  const WorkItem it = p.items[blockIdx.x];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane / LPR, dl = lane % LPR;
  const int tmask = (dl >> TB) & 7;              // token permutation of this lane
  const int Q = p.Q;
  const int b = p.virt ? it.unit / Q : it.unit;
  const int qi = p.virt ? it.unit % Q : 0;
  const int len = p.units[it.unit].len;          // keys visible to this unit
  const int kvh = it.kvh;
  const int Hkv = p.kv.hkv;

  // ---- query slice in registers, pre-scaled
  float2 q2[R][4];
  {
    float qs = p.scale_log2 * (has_global_scale(DT) ? p.kv.kg : 1.0f);
    const __nv_bfloat16 *qb = p.q + (((size_t)b * Q + qi) * p.Hq + (size_t)kvh * p.G) * D + dl * 8;
#pragma unroll
    for (int h = 0; h < R; ++h) {
      uint4 u = *reinterpret_cast<const uint4 *>(qb + (size_t)h * D);
      float2 f0 = bf16x2_to_f2(u.x), f1 = bf16x2_to_f2(u.y), f2 = bf16x2_to_f2(u.z),
             f3 = bf16x2_to_f2(u.w);
      q2[h][0] = make_float2(f0.x * qs, f0.y * qs);
      q2[h][1] = make_float2(f1.x * qs, f1.y * qs);
      q2[h][2] = make_float2(f2.x * qs, f2.y * qs);
      q2[h][3] = make_float2(f3.x * qs, f3.y * qs);
    }
  }

  // ---- this warp's iterations
  const int t_begin = it.blk_begin * kBlock;
  const int t_end = min(len, it.blk_end * kBlock);
  const int n_it = t_end > t_begin ? (t_end - t_begin + TOK - 1) / TOK : 0;
  const int n_local = n_it > warp ? (n_it - warp + kWarps - 1) / kWarps : 0;

  uint8_t *wsm = smem + warp * Gm::WARP_BYTES;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int *trow = p.tables + (size_t)b * p.stride;
  const uint64_t pol = policy_evict_first();
  int tab_cache = -1, tab_chunk = -1;
  uint32_t valid_bits = 0;   // stage validity (bit s)
  bool failed = false;

  // issue the copies of local iteration j into its stage (all lanes call)
  auto issue = [&](int j) {
    const int k = warp + j * kWarps;                 // iteration within the item
    const int blk = it.blk_begin + k / IPB;
    const int sub = k % IPB;
    const int chunk = j >> 5;
    if (chunk != tab_chunk) {
      const int jj = chunk * 32 + lane;
      const int kk = warp + jj * kWarps;
      tab_cache = (jj < n_local) ? __ldg(trow + it.blk_begin + kk / IPB) : -1;
      tab_chunk = chunk;
    }
    const int phys = __shfl_sync(0xffffffffu, tab_cache, j & 31);
    const int s = j % NSTAGE;
    const bool ok = phys >= 0 && phys < p.kv.num_blocks;
    valid_bits = ok ? (valid_bits | (1u << s)) : (valid_bits & ~(1u << s));
    if (lane == 0) {
      uint64_t *bar = &bars[warp][s];
      if (!ok) {
        set_err(p.hdr, PA_ERRF_BAD_BLOCK_ID);
        mbar_arrive(bar);
      } else {
        uint8_t *st = wsm + s * Gm::STAGE;
        const size_t tile = (size_t)phys * Hkv + kvh;
        const size_t code_off = tile * kBlock * Gm::ROW_BYTES + (size_t)sub * Gm::CODE_BYTES;
        uint32_t bytes = 2 * Gm::CODE_BYTES;
        if constexpr (has_scale_tensors(DT)) bytes += 2 * Gm::SCALE_BYTES;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(st, (const uint8_t *)p.kv.k + code_off, Gm::CODE_BYTES, bar, pol);
        bulk_g2s(st + Gm::CODE_BYTES, (const uint8_t *)p.kv.v + code_off, Gm::CODE_BYTES, bar, pol);
        if constexpr (has_scale_tensors(DT)) {
          const size_t sc_off = tile * kBlock * Gm::SROW_BYTES + (size_t)sub * Gm::SCALE_BYTES;
          bulk_g2s(st + 2 * Gm::CODE_BYTES, (const uint8_t *)p.kv.ks + sc_off, Gm::SCALE_BYTES, bar,
                   pol);
          bulk_g2s(st + 2 * Gm::CODE_BYTES + Gm::SCALE_BYTES, (const uint8_t *)p.kv.vs + sc_off,
                   Gm::SCALE_BYTES, bar, pol);
        }
      }
    }
  };

  // ---- softmax state
  float m_run[R];
  float l_part[NH];
  float2 o2[R][4];
#pragma unroll
  for (int h = 0; h < R; ++h) {
    m_run[h] = kNegInf;
#pragma unroll
    for (int j = 0; j < 4; ++j) o2[h][j] = make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int h = 0; h < NH; ++h) l_part[h] = 0.f;

  // lane bits used by the head steps
  const int hb1 = SPLIT1 ? ((lane >> (TB - 1)) & 1) : 0;
  int hbase = 0;
  if constexpr (TB >= 1 && SPLIT1) hbase += hb1 * (R / 2);
  if constexpr (TB >= 2 && SPLIT2) hbase += (lane & 1) * (N1 / 2);
  int dupmask = 0;
  if constexpr (TB >= 1 && !SPLIT1) dupmask |= 1 << (TB - 1);
  if constexpr (TB >= 2 && !SPLIT2) dupmask |= 1;
  const bool owner = (lane & dupmask) == 0;

  const int prologue = min(NSTAGE, n_local);
  for (int j = 0; j < prologue; ++j) issue(j);
  int issued = prologue;

  for (int j = 0; j < n_local; ++j) {
    const int s = j % NSTAGE;
    const bool arrived = mbar_wait(&bars[warp][s], (j / NSTAGE) & 1);
    if (!__all_sync(0xffffffffu, arrived)) {   // warp-uniform decision
      failed = true;
      if (lane == 0) set_err(p.hdr, PA_ERRF_WAIT_TIMEOUT);
      break;
    }
    const int k = warp + j * kWarps;
    const int tok0 = t_begin + k * TOK;              // first token of this iteration
    if (valid_bits & (1u << s)) {
      const uint8_t *st = wsm + s * Gm::STAGE;
      const uint8_t *sK = st, *sV = st + Gm::CODE_BYTES;
      const uint8_t *sKs = st + 2 * Gm::CODE_BYTES, *sVs = sKs + Gm::SCALE_BYTES;

      // ---- partial scores: 8 tokens (XOR-permuted) x R heads over this lane's slice
      float a[8][R];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float2 kf[4];
        load8<DT, D>(sK, sKs, rg * 8 + (r ^ tmask), dl, kf);
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float2 acc = fmul2(q2[h][0], kf[0]);
          acc = ffma2(q2[h][1], kf[1], acc);
          acc = ffma2(q2[h][2], kf[2], acc);
          acc = ffma2(q2[h][3], kf[3], acc);
          a[r][h] = acc.x + acc.y;
        }
      }
      // token steps (reduce-scatter over the 8 lanes sharing the low bits)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int h = 0; h < R; ++h) a[r][h] += __shfl_xor_sync(0xffffffffu, a[r + 4][h], 4 << TB);
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < R; ++h) a[r][h] += __shfl_xor_sync(0xffffffffu, a[r + 2][h], 2 << TB);
#pragma unroll
      for (int h = 0; h < R; ++h) a[0][h] += __shfl_xor_sync(0xffffffffu, a[1][h], 1 << TB);
      // head steps
      float sc[R];
#pragma unroll
      for (int h = 0; h < R; ++h) sc[h] = a[0][h];
      if constexpr (TB >= 1) {
        constexpr int dist = 1 << (TB - 1);
        if constexpr (SPLIT1) {
#pragma unroll
          for (int h = 0; h < R / 2; ++h) {
            float mine = hb1 ? sc[h + R / 2] : sc[h];
            float other = hb1 ? sc[h] : sc[h + R / 2];
            sc[h] = mine + __shfl_xor_sync(0xffffffffu, other, dist);
          }
        } else {
#pragma unroll
          for (int h = 0; h < R; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], dist);
        }
      }
      if constexpr (TB >= 2) {
        const int hb2 = lane & 1;
        if constexpr (SPLIT2) {
#pragma unroll
          for (int h = 0; h < N1 / 2; ++h) {
            float mine = hb2 ? sc[h + N1 / 2] : sc[h];
            float other = hb2 ? sc[h] : sc[h + N1 / 2];
            sc[h] = mine + __shfl_xor_sync(0xffffffffu, other, 1);
          }
        } else {
#pragma unroll
          for (int h = 0; h < N1; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], 1);
        }
      }
      // this lane now holds heads [hbase, hbase + NH) of token tl
      const int tl = rg * 8 + tmask;
      const bool tvalid = tok0 + tl < t_end;
      float kscale = 1.f;
      if constexpr (DT == PA_KV_INT8)
        kscale = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sKs)[tl]);
      float s_[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) s_[h] = tvalid ? sc[h] * kscale : kNegInf;

      // max over the iteration's tokens for the held heads
      float mx[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float v = s_[h];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1 << TB));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2 << TB));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4 << TB));
        if constexpr (RG == 2) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mx[h] = v;
      }
      if (tmask == 0 && rg == 0 && owner) {
#pragma unroll
        for (int h = 0; h < NH; ++h) red[warp][hbase + h] = mx[h];
      }
      __syncwarp();
      bool need = false;
      float mrow[R];
#pragma unroll
      for (int h = 0; h < R; ++h) {
        mrow[h] = red[warp][h];
        need |= mrow[h] > m_run[h] + kRescale;
      }
      if (need) {   // warp-uniform
        float alpha[R];
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float mn = fmaxf(m_run[h], mrow[h]);
          alpha[h] = (mn == kNegInf) ? 1.f : exp2f(m_run[h] - mn);
          m_run[h] = mn;
#pragma unroll
          for (int j2 = 0; j2 < 4; ++j2) {
            o2[h][j2].x *= alpha[h];
            o2[h][j2].y *= alpha[h];
          }
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float al = alpha[h];
#pragma unroll
          for (int c = 1; c < R / NH; ++c)
            if (hbase == c * NH) al = alpha[c * NH + h];
          l_part[h] *= al;
        }
      }
      // probabilities for the held (token, heads)
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float mh = m_run[h];
#pragma unroll
        for (int c = 1; c < R / NH; ++c)
          if (hbase == c * NH) mh = m_run[c * NH + h];
        float pr = (s_[h] == kNegInf) ? 0.f : exp2f(s_[h] - mh);
        l_part[h] += pr;
        s_[h] = pr;
      }
      if (owner) {
#pragma unroll
        for (int h = 0; h < NH; ++h) pbuf[warp][tl][hbase + h] = s_[h];
      }
      __syncwarp();
      // ---- PV over this row group's tokens
#pragma unroll 2
      for (int t = rg * 8; t < rg * 8 + 8; ++t) {
        if (tok0 + t >= t_end) break;
        float2 vf[4];
        load8<DT, D>(sV, sVs, t, dl, vf);
        float4 pa4 = *reinterpret_cast<const float4 *>(&pbuf[warp][t][0]);
        float4 pb4 = *reinterpret_cast<const float4 *>(&pbuf[warp][t][4]);
        float pp[8] = {pa4.x, pa4.y, pa4.z, pa4.w, pb4.x, pb4.y, pb4.z, pb4.w};
        if constexpr (DT == PA_KV_INT8) {
          float vs = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sVs)[t]);
#pragma unroll
          for (int h = 0; h < R; ++h) pp[h] *= vs;
        }
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float2 ph = make_float2(pp[h], pp[h]);
#pragma unroll
          for (int j2 = 0; j2 < 4; ++j2) o2[h][j2] = ffma2(ph, vf[j2], o2[h][j2]);
        }
      }
    }
    __syncwarp();
    if (issued < n_local) {
      issue(issued);
      ++issued;
    }
  }
  if (failed) {   // let copies still in flight land before the stages are reused
    // (only the last fill of each stage can be in flight; an older phase's
    // parity repeats and would read as pending)
    for (int j = max(issued - NSTAGE, 0); j < issued; ++j)
      (void)mbar_wait(&bars[warp][j % NSTAGE], (j / NSTAGE) & 1);
  }

  // ---- per-warp totals: l over lanes, o over row groups
  float lsum[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    float v = owner ? l_part[h] : 0.f;
    v += __shfl_xor_sync(0xffffffffu, v, 1 << TB);
    v += __shfl_xor_sync(0xffffffffu, v, 2 << TB);
    v += __shfl_xor_sync(0xffffffffu, v, 4 << TB);
    if constexpr (RG == 2) v += __shfl_xor_sync(0xffffffffu, v, 16);
    lsum[h] = v;
  }
  if constexpr (RG == 2) {
#pragma unroll
    for (int h = 0; h < R; ++h)
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        o2[h][j2].x += __shfl_xor_sync(0xffffffffu, o2[h][j2].x, 16);
        o2[h][j2].y += __shfl_xor_sync(0xffffffffu, o2[h][j2].y, 16);
      }
  }
  if (tmask == 0 && rg == 0 && owner) {
#pragma unroll
    for (int h = 0; h < NH; ++h) s_l[warp][hbase + h] = lsum[h];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < R; ++h) s_m[warp][h] = m_run[h];
  }
  // this warp's o goes into its own (now idle) stage area
  float *ow = reinterpret_cast<float *>(wsm);
  if (rg == 0) {
#pragma unroll
    for (int h = 0; h < R; ++h) {
      float4 *dst = reinterpret_cast<float4 *>(ow + h * D + dl * 8);
      dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
      dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
    }
  }
  __syncthreads();

  // ---- merge the warps and write
  const float vg = has_global_scale(DT) ? p.kv.vg : 1.0f;
  const int G = p.G;
  for (int idx = threadIdx.x; idx < R * D; idx += kThreads) {
    const int h = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      float mw = s_m[w][h];
      float f = (mw == kNegInf) ? 0.f : exp2f(mw - M);
      L += f * s_l[w][h];
      acc += f * reinterpret_cast<const float *>(smem + w * Gm::WARP_BYTES)[h * D + d];
    }
    const float o = L > 0.f ? acc / L * vg : 0.f;
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : kNegInf;
    if (it.parts <= 1) {
      const size_t row = ((size_t)b * Q + qi) * p.Hq + (size_t)kvh * G + h;
      if (p.out_fp32)
        reinterpret_cast<float *>(p.out)[row * D + d] = o;
      else
        reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(o);
      if (d == 0 && p.lse_out) p.lse_out[row] = lse;
    } else {
      const size_t prow = ((size_t)it.slot * Hkv + kvh) * R + h;
      p.part_o[prow * D + d] = o;
      if (d == 0) p.part_lse[prow] = lse;
    }
  }
}

template <int DT, int D, int R>
cudaError_t launch_one(const AttnParams &p, int grid, cudaStream_t s) {
  using Gm = Geo<DT, D>;
  auto kern = decode_kernel<DT, D, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, kThreads, Gm::SMEM, s, p);
}

template <int DT>
cudaError_t launch_dtype(const AttnParams &p, int grid, cudaStream_t s) {
  const int D = p.kv.D, R = p.R;
#define PA_SIMT_CASE(DD, RR) \
  if (D == DD && R == RR) return launch_one<DT, DD, RR>(p, grid, s);
  PA_SIMT_CASE(128, 1) PA_SIMT_CASE(128, 2) PA_SIMT_CASE(128, 4) PA_SIMT_CASE(128, 6)
  PA_SIMT_CASE(128, 8) PA_SIMT_CASE(256, 1) PA_SIMT_CASE(256, 2) PA_SIMT_CASE(256, 4)
  PA_SIMT_CASE(256, 6) PA_SIMT_CASE(256, 8)
#undef PA_SIMT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace simt
}  // namespace pa
