// pa_verify_mma.cuh -- speculative verify as dense tensor-core tiles per
// (sequence, row group, kv head, key range): the Q query tokens x G heads
// rows share every key block; groups hold up to 48 rows (beyond that the
// planner keeps a sequence's groups adjacent so their key reads hit L2).
// The scores S^T [16 tokens x R] = K Q^T and the
// update O^T [D x R] += V^T P^T are dense contractions ("vLLM All-NVFP4
// DFlash2 for Blackwell", "What makes this stack different": DFlash2 K=7, 8
// query tokens per verify step; causal among the new tokens: the virtual
// batch of "vLLM-SM70", "Why", where query i sees keys t < L - Q + 1 + i).
//
// One CTA of 4 warps walks the item's 16-token blocks together; the KV
// codes of a block arrive once (TMA, 128-byte swizzle) and each warp owns a
// 64-wide slice of the head dim:
//   1. QK: the warp dequantises its slice of K and computes partial scores
//      for all R rows (mma.sync m16n8k16, f16 operands, fp32 accumulation).
//   2. The partials go through shared memory once; warp o finishes the
//      columns whose fragment pair index is o (a reduce-scatter), applies
//      scales, the causal mask and the online softmax (log2 domain, lazy
//      rescale), and writes P as f16 in a layout the B fragments read with
//      one 8-byte load per n-tile.
//   3. PV: the warp dequantises its slice of V and accumulates O^T for all
//      R rows over its 64 head-dim rows.
// Every K and V element is dequantised exactly once, which is what the
// per-query virtual batch cannot do.
#pragma once

#include "pa_decode_mma.cuh"

namespace pa {
namespace vfy {

using tc::e2m1x8_to_h2x4;
using tc::e4m3x2_to_h2;
using tc::ex2f;
using tc::f2_to_h2;
using tc::mma16816;
using tc::prmt;
using tc::s8pair_to_h2;
using tc::sw_off;
using tc::tma_rows;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int D = 256;
constexpr int DS = D / kWarps;   // head-dim slice per warp

template <int DT, int NT>
struct Geo {
  static_assert(DT == PA_KV_INT8 || DT == PA_KV_NVFP4 || DT == PA_KV_FP8, "quantised formats");
  static_assert(NT % 2 == 0 && NT <= 6, "even n-tile count");
  static constexpr int ROW = DT == PA_KV_NVFP4 ? D / 2 : D;
  static constexpr int SROW = DT == PA_KV_INT8 ? 2 : (DT == PA_KV_NVFP4 ? D / 16 : 0);
  static constexpr int CODE = kBlock * ROW;
  static constexpr int SC = kBlock * SROW;
  static constexpr int PAYLOAD = 2 * (CODE + SC);
  static constexpr int STAGE = (PAYLOAD + 1023) / 1024 * 1024;
  static constexpr int NSTAGE = 8;
  static constexpr int NC = 8 * NT;                       // columns (rows of Q)
  static constexpr int EPO = NT / 2;                      // entries per owner lane per token
  // partial scores [src warp][token][owner][EST]: EST = 2 NT + 2 floats makes
  // the 16 float2 stores of a half-warp hit 32 distinct banks
  static constexpr int EST = 2 * NT + 2;
  static constexpr int SBUF = kWarps * kBlock * kWarps * EST * 4;
  static constexpr int PBUF = NC * kBlock * 2;            // P, f16 [col][16 tokens]
  static constexpr int SMEM = NSTAGE * STAGE + SBUF + PBUF + 1024;
};

template <int DT, int NT>
__global__ void __launch_bounds__(kThreads, NT == 2 ? 4 : 2)
    verify_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using Gm = Geo<DT, NT>;
  constexpr int NSTAGE = Gm::NSTAGE, ROW = Gm::ROW, SROW = Gm::SROW, NC = Gm::NC, EPO = Gm::EPO;
  constexpr float kRescale = 8.0f;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *stages = smem;
  float *sbuf = reinterpret_cast<float *>(smem + NSTAGE * Gm::STAGE);
  uint16_t *pbuf = reinterpret_cast<uint16_t *>(smem + NSTAGE * Gm::STAGE + Gm::SBUF);
  __shared__ __align__(8) uint64_t bars[NSTAGE];
  __shared__ float s_alpha[NC];
  __shared__ float s_l[NC], s_m[NC];
  __shared__ int s_fail;

  griddep_launch();   // the merge may start launching once every CTA has begun
  griddep_wait();     // the plan of this call is complete
  const uint32_t num_items = p.hdr[HDR_NUM_ITEMS];
  if (blockIdx.x >= num_items) return;
  const WorkItem it = p.items[blockIdx.x];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  // unit = (sequence, row group): rows ro .. ro + R - 1 of the sequence's Q * G
  const int b = it.unit / p.RG, ro = (it.unit % p.RG) * p.R;
  const int kvh = it.kvh, Q = p.Q, G = p.G, Hkv = p.kv.hkv;
  const int R = min(p.R, Q * G - ro);   // live rows of this group
  const int L = p.units[it.unit].len;   // keys of the sequence (the last row's limit)

  // ---- Q fragments of this warp's head-dim slice, all n-tiles
  uint32_t qf[NT][4][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = nt * 8 + r;
    const bool live = n < R;
    const int qi = live ? (ro + n) / G : 0, g = live ? (ro + n) % G : 0;
    const __nv_bfloat16 *qrow = p.q + (((size_t)b * Q + qi) * p.Hq + (size_t)kvh * G + g) * D;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int d = warp * DS + c * 16 + 4 * s;
      uint2 u = live ? *reinterpret_cast<const uint2 *>(qrow + d) : make_uint2(0, 0);
      float2 x0 = bf16x2_to_f2(u.x), x1 = bf16x2_to_f2(u.y);
      qf[nt][s][0] = f2_to_h2(x0.x, x0.y);
      qf[nt][s][1] = f2_to_h2(x1.x, x1.y);
    }
  }
  const float qscale = p.scale_log2 * (has_global_scale(DT) ? p.kv.kg : 1.0f);

  // owner side: this lane finishes entries e = c*EPO + k (k < EPO) of every
  // token pair (r, r+8) in warp `warp`'s column set: column = (e/2)*8 + 2*warp + e%2
  int ocol[EPO], olim[EPO];
#pragma unroll
  for (int k = 0; k < EPO; ++k) {
    const int e = c * EPO + k;
    ocol[k] = (e >> 1) * 8 + 2 * warp + (e & 1);
    const int qi = (ro + ocol[k]) / G;
    olim[k] = ocol[k] < R ? L - Q + 1 + qi : 0;   // keys visible to that query row
  }
  float m_run[EPO], l_run[EPO];
#pragma unroll
  for (int k = 0; k < EPO; ++k) {
    m_run[k] = kNegInf;
    l_run[k] = 0.f;
  }
  float o[4][NT][4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[e][nt][k] = 0.f;

  const int t_begin = it.blk_begin * kBlock;
  const int t_end = min(L, it.blk_end * kBlock);
  const int n_blk = t_end > t_begin ? (t_end - t_begin + kBlock - 1) / kBlock : 0;
  const int *trow = p.tables + (size_t)b * p.stride;
  const uint64_t pol = policy_evict_first();

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    s_fail = 0;
  }
  __syncthreads();
  uint32_t valid_bits = 0;   // tracked by thread 0 only, broadcast through s_valid
  __shared__ uint32_t s_valid;

  // thread 0 issues block j; its table entry was loaded one issue earlier
  int next_phys = (tid == 0 && n_blk > 0) ? trow[it.blk_begin] : -1;
  auto issue = [&](int j) {   // thread 0
    const int s = j % NSTAGE;
    const int phys = next_phys;
    if (j + 1 < n_blk) next_phys = trow[it.blk_begin + j + 1];   // consumed next time
    const bool ok = phys >= 0 && phys < p.kv.num_blocks;
    valid_bits = ok ? (valid_bits | (1u << s)) : (valid_bits & ~(1u << s));
    uint64_t *bar = &bars[s];
    if (!ok) {
      set_err(p.hdr, PA_ERRF_BAD_BLOCK_ID);
      mbar_arrive(bar);
      return;
    }
    uint8_t *st = stages + s * Gm::STAGE;
    const size_t tile = (size_t)phys * Hkv + kvh;
    const int y = (int)(tile * kBlock);
    mbar_arrive_expect_tx(bar, Gm::PAYLOAD);
#pragma unroll
    for (int x = 0; x < ROW; x += 128) {
      tma_rows(st + x * kBlock, &tmK, x, y, bar, pol);
      tma_rows(st + Gm::CODE + x * kBlock, &tmV, x, y, bar, pol);
    }
    if constexpr (Gm::SC > 0) {
      bulk_g2s(st + 2 * Gm::CODE, (const uint8_t *)p.kv.ks + tile * Gm::SC, Gm::SC, bar, pol);
      bulk_g2s(st + 2 * Gm::CODE + Gm::SC, (const uint8_t *)p.kv.vs + tile * Gm::SC, Gm::SC, bar,
               pol);
    }
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < min(NSTAGE, n_blk); ++issued) issue(issued);
    s_valid = valid_bits;
  }
  __syncthreads();   // s_valid of the first NSTAGE blocks visible

  for (int j = 0; j < n_blk; ++j) {
    const int s = j % NSTAGE;
    const bool arrived = mbar_wait(&bars[s], (j / NSTAGE) & 1);
    const bool valid = arrived && ((s_valid >> s) & 1u);
    const uint8_t *st = stages + s * Gm::STAGE;
    const uint8_t *sK = st, *sV = st + Gm::CODE, *sKs = st + 2 * Gm::CODE, *sVs = sKs + Gm::SC;
    const int tok0 = t_begin + j * kBlock;
    const int nvalid = min(kBlock, t_end - tok0);

    // ---- 1. partial scores over this warp's head-dim slice
    float sp[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) sp[nt][k] = 0.f;
    if (valid) {
      if constexpr (DT == PA_KV_NVFP4) {
        const int kb = warp * (DS / 2) + c * 8;   // 8 bytes = 16 elements of row r
        uint2 k0 = *reinterpret_cast<const uint2 *>(sK + sw_off(r, kb));
        uint2 k1 = *reinterpret_cast<const uint2 *>(sK + sw_off(r, kb) + 8 * 128);
        const uint32_t sa = e4m3_to_h2_dup(sKs[r * SROW + warp * 4 + c]);
        const uint32_t sb = e4m3_to_h2_dup(sKs[(r + 8) * SROW + warp * 4 + c]);
        uint32_t w0[2] = {k0.x, k0.y}, w1[2] = {k1.x, k1.y};
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          uint32_t h0[4], h1[4];
          e2m1x8_to_h2x4(w0[wi], h0);
          e2m1x8_to_h2x4(w1[wi], h1);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t a0 = hmul2_u32(h0[2 * hh], sa), a1 = hmul2_u32(h1[2 * hh], sb);
            const uint32_t a2 = hmul2_u32(h0[2 * hh + 1], sa), a3 = hmul2_u32(h1[2 * hh + 1], sb);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816(sp[nt], a0, a1, a2, a3, qf[nt][2 * wi + hh][0], qf[nt][2 * wi + hh][1]);
          }
        }
      } else {
        const int kb = warp * DS + c * 16;   // 16 bytes = 16 codes of row r
        uint4 k0 = *reinterpret_cast<const uint4 *>(sK + sw_off(r, kb));
        uint4 k1 = *reinterpret_cast<const uint4 *>(sK + sw_off(r, kb) + 8 * 128);
        uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
          uint32_t a0, a1, a2, a3;
          if constexpr (DT == PA_KV_INT8) {
            const uint32_t x0 = w0[s2] ^ 0x80808080u, x1 = w1[s2] ^ 0x80808080u;
            a0 = s8pair_to_h2(x0, 0);
            a1 = s8pair_to_h2(x1, 0);
            a2 = s8pair_to_h2(x0, 1);
            a3 = s8pair_to_h2(x1, 1);
          } else {   // FP8: bytes 0,1 -> k rows 2c, 2c+1; bytes 2,3 -> 2c+8, 2c+9
            a0 = e4m3x2_u16_to_h2(w0[s2]);
            a1 = e4m3x2_u16_to_h2(w1[s2]);
            a2 = e4m3x2_u16_to_h2(w0[s2] >> 16);
            a3 = e4m3x2_u16_to_h2(w1[s2] >> 16);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma16816(sp[nt], a0, a1, a2, a3, qf[nt][s2][0], qf[nt][s2][1]);
        }
      }
    }
    // ---- 2. reduce-scatter the partials: owner of column pair index c is warp c
    {
      constexpr int EST = Gm::EST;
      float *dst0 = sbuf + (((warp * kBlock + r) * kWarps + c) * EST);
      float *dst1 = sbuf + (((warp * kBlock + r + 8) * kWarps + c) * EST);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        *reinterpret_cast<float2 *>(dst0 + 2 * nt) = make_float2(sp[nt][0], sp[nt][1]);
        *reinterpret_cast<float2 *>(dst1 + 2 * nt) = make_float2(sp[nt][2], sp[nt][3]);
      }
    }
    if (__syncthreads_or(!arrived)) {   // B1: partials visible; every thread is past block j-1
      if (tid == 0) set_err(p.hdr, PA_ERRF_WAIT_TIMEOUT);
      s_fail = 1;
      break;
    }
    // block j-1's stage is consumed by everyone: refill it with block j-1+NSTAGE
    if (tid == 0 && j >= 1 && issued < n_blk) {
      issue(issued);
      ++issued;
      s_valid = valid_bits;
    }
    float sc[EPO][2];
#pragma unroll
    for (int k = 0; k < EPO; ++k) {
      const int e = c * EPO + k;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        a0 += sbuf[((w * kBlock + r) * kWarps + warp) * Gm::EST + e];
        a1 += sbuf[((w * kBlock + r + 8) * kWarps + warp) * Gm::EST + e];
      }
      sc[k][0] = a0;
      sc[k][1] = a1;
    }
    float f0 = qscale, f1 = qscale;
    if constexpr (DT == PA_KV_INT8) {
      f0 *= fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sKs)[r]);
      f1 *= fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sKs)[r + 8]);
    }
    bool need = false;
    float mx[EPO];
#pragma unroll
    for (int k = 0; k < EPO; ++k) {
      const bool ok0 = valid && r < nvalid && tok0 + r < olim[k];
      const bool ok1 = valid && r + 8 < nvalid && tok0 + r + 8 < olim[k];
      sc[k][0] = ok0 ? sc[k][0] * f0 : kNegInf;
      sc[k][1] = ok1 ? sc[k][1] * f1 : kNegInf;
      // the lane's own scores decide whether the running max must move; only
      // then is the column max reduced over the 8 lanes holding the column
      mx[k] = fmaxf(sc[k][0], sc[k][1]);
      need |= mx[k] > m_run[k] + kRescale;
    }
    const bool any_need = __syncthreads_or(need);   // B2
    if (any_need) {
#pragma unroll
      for (int k = 0; k < EPO; ++k) {
        float v = mx[k];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        const float mn = fmaxf(m_run[k], v);
        const float al = (mn == kNegInf) ? 1.f : ex2f(m_run[k] - mn);
        m_run[k] = mn;
        l_run[k] *= al;
        if (r == 0) s_alpha[ocol[k]] = al;
      }
    }
    // probabilities -> P (f16) at [column][token slot]; token 2c'+{0,1} at slot
    // 4c'+{0,1}, token 2c'+8+{0,1} at slot 4c'+2+{0,1}
    {
      const int slot0 = (r >> 1) * 4 + (r & 1), slot1 = slot0 + 2;
      float vs0 = 1.f, vs1 = 1.f;
      if constexpr (DT == PA_KV_INT8) {
        vs0 = (valid && r < nvalid) ? fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sVs)[r]) : 0.f;
        vs1 = (valid && r + 8 < nvalid) ? fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sVs)[r + 8])
                                        : 0.f;
      }
#pragma unroll
      for (int k = 0; k < EPO; ++k) {
        const float p0 = sc[k][0] == kNegInf ? 0.f : ex2f(sc[k][0] - m_run[k]);
        const float p1 = sc[k][1] == kNegInf ? 0.f : ex2f(sc[k][1] - m_run[k]);
        l_run[k] += p0 + p1;
        const __half h0 = __float2half_rn(p0 * vs0), h1 = __float2half_rn(p1 * vs1);
        pbuf[ocol[k] * kBlock + slot0] = __half_as_ushort(h0);
        pbuf[ocol[k] * kBlock + slot1] = __half_as_ushort(h1);
      }
    }
    __syncthreads();   // B3: P and alphas visible
    // ---- 3. PV over this warp's head-dim slice
    if (any_need) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float a0 = s_alpha[nt * 8 + 2 * c], a1 = s_alpha[nt * 8 + 2 * c + 1];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[e][nt][0] *= a0;
          o[e][nt][1] *= a1;
          o[e][nt][2] *= a0;
          o[e][nt][3] *= a1;
        }
      }
    }
    if (valid) {
      uint32_t B[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint2 u = *reinterpret_cast<const uint2 *>(pbuf + (nt * 8 + r) * kBlock + c * 4);
        B[nt][0] = u.x;
        B[nt][1] = u.y;
      }
      const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
      if constexpr (DT == PA_KV_NVFP4) {
        const int vb = warp * (DS / 2) + r * 4;   // 4 bytes = 8 elements
        uint32_t vw[4], vsb[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool ok = tk[t] < nvalid;
          vw[t] = ok ? *reinterpret_cast<const uint32_t *>(sV + sw_off(tk[t], vb)) : 0u;
          vsb[t] = ok ? sVs[tk[t] * SROW + warp * 4 + (r >> 1)] : 0u;
        }
        const uint32_t spa = e4m3x2_to_h2(vsb[0], vsb[1]), spb = e4m3x2_to_h2(vsb[2], vsb[3]);
        uint32_t xa[4], ya[4], xb[4], yb[4];
        e2m1x8_to_h2x4((vw[0] & 0x0F0F0F0Fu) | ((vw[1] << 4) & 0xF0F0F0F0u), xa);
        e2m1x8_to_h2x4(((vw[0] >> 4) & 0x0F0F0F0Fu) | (vw[1] & 0xF0F0F0F0u), ya);
        e2m1x8_to_h2x4((vw[2] & 0x0F0F0F0Fu) | ((vw[3] << 4) & 0xF0F0F0F0u), xb);
        e2m1x8_to_h2x4(((vw[2] >> 4) & 0x0F0F0F0Fu) | (vw[3] & 0xF0F0F0F0u), yb);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t a0 = hmul2_u32(xa[e], spa), a1 = hmul2_u32(ya[e], spa);
          const uint32_t a2 = hmul2_u32(xb[e], spb), a3 = hmul2_u32(yb[e], spb);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(o[e][nt], a0, a1, a2, a3, B[nt][0], B[nt][1]);
        }
      } else {
        const int vb = warp * DS + r * 8;   // 8 bytes = 8 codes
        uint32_t vw[4][2];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool ok = tk[t] < nvalid;
          uint2 u = ok ? *reinterpret_cast<const uint2 *>(sV + sw_off(tk[t], vb)) : make_uint2(0, 0);
          const uint32_t flip = DT == PA_KV_INT8 ? 0x80808080u : 0u;   // int8: offset-binary
          vw[t][0] = u.x ^ flip;
          vw[t][1] = u.y ^ flip;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a0, a1, a2, a3;
          if constexpr (DT == PA_KV_INT8) {
            uint32_t h[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) h[t] = s8pair_to_h2(vw[t][e >> 1], e & 1);
            a0 = prmt(h[0], h[1], 0x5410);
            a1 = prmt(h[0], h[1], 0x7632);
            a2 = prmt(h[2], h[3], 0x5410);
            a3 = prmt(h[2], h[3], 0x7632);
          } else {   // FP8: interleave the bytes of each token pair, one cvt per register
            const uint32_t sel = (e & 1) ? 0x7362u : 0x5140u;
            const uint32_t xa = prmt(vw[0][e >> 1], vw[1][e >> 1], sel);
            const uint32_t xb = prmt(vw[2][e >> 1], vw[3][e >> 1], sel);
            a0 = e4m3x2_u16_to_h2(xa);
            a1 = e4m3x2_u16_to_h2(xa >> 16);
            a2 = e4m3x2_u16_to_h2(xb);
            a3 = e4m3x2_u16_to_h2(xb >> 16);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(o[e][nt], a0, a1, a2, a3, B[nt][0], B[nt][1]);
        }
      }
    }
    // block j+1's B1 orders these reads of stage s and of P before stage s is
    // refilled and before P is rewritten
  }
  if (s_fail && tid == 0) {   // only the last fill of each stage can be in flight
    for (int j = max(issued - NSTAGE, 0); j < issued; ++j)
      (void)mbar_wait(&bars[j % NSTAGE], (j / NSTAGE) & 1);
  }

  // ---- finish: row sums and max per column, then O / l
#pragma unroll
  for (int k = 0; k < EPO; ++k) {
    float v = l_run[k];
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    if (r == 0) {
      s_l[ocol[k]] = v;
      s_m[ocol[k]] = m_run[k];
    }
  }
  __syncthreads();
  const float vg = has_global_scale(DT) ? p.kv.vg : 1.0f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int n = nt * 8 + 2 * c + jj;
      if (n >= R) continue;
      const float Lr = s_l[n];
      const float inv = Lr > 0.f ? vg / Lr : 0.f;
      const int qi = (ro + n) / G, g = (ro + n) % G;
      const size_t orow = ((size_t)b * Q + qi) * p.Hq + (size_t)kvh * G + g;
      const size_t prow = ((size_t)it.slot * Hkv + kvh) * p.R + n;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = warp * DS + r * 8 + 2 * e;
        const float x0 = o[e][nt][jj] * inv, x1 = o[e][nt][2 + jj] * inv;
        if (it.parts <= 1) {
          if (p.out_fp32)
            *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.out) + orow * D + d) =
                make_float2(x0, x1);
          else
            *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * D +
                                                d) = __floats2bfloat162_rn(x0, x1);
        } else {
          *reinterpret_cast<float2 *>(p.part_o + prow * D + d) = make_float2(x0, x1);
        }
      }
      if (warp == 0 && r == 0) {
        const float lse = Lr > 0.f ? (s_m[n] + __log2f(Lr)) * 0.69314718055994531f : kNegInf;
        if (it.parts <= 1) {
          if (p.lse_out) p.lse_out[orow] = lse;
        } else {
          p.part_lse[prow] = lse;
        }
      }
    }
}

template <int DT, int NT>
cudaError_t launch_one(const AttnParams &p, int grid, cudaStream_t s) {
  using Gm = Geo<DT, NT>;
  auto kern = verify_kernel<DT, NT>;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)p.kv.num_blocks * p.kv.hkv * kBlock;
  if (!tc::make_row_map(&tk, p.kv.k, Gm::ROW, rows) || !tc::make_row_map(&tv, p.kv.v, Gm::ROW, rows))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, kThreads, Gm::SMEM, s, p, tk, tv);
}

template <int DT>
cudaError_t launch_dtype(const AttnParams &p, int grid, cudaStream_t s) {
  switch (p.R) {   // rows per group -> n-tiles of 8 columns
    case 16: return launch_one<DT, 2>(p, grid, s);
    case 32: return launch_one<DT, 4>(p, grid, s);
    case 48: return launch_one<DT, 6>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vfy
}  // namespace pa
