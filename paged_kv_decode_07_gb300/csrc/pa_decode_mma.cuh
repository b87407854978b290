// pa_decode_mma.cuh -- split-K paged decode attention on the tensor cores
// (mma.sync m16n8k16, fp32 accumulation) for every KV format: f16 operands
// dequantised from the int8, NVFP4 and FP8-E4M3 codes, bf16 operands read
// straight from bf16 KV.
//
// Why tensor cores for decode: with GQA the G query heads of one kv head
// share every key and value, so per (token, kv head) the scores and the PV
// update are a dense [G x D] x [D x 16-token] contraction -- 3,072 FMA per
// token and kv head at D = 256, G = 6.  Against 516 B (int8) or 288 B
// (NVFP4) per token and kv head that is 11.9 / 21.3 FLOP per byte, more
// than the CUDA cores can issue next to the dequant at HBM speed (the
// counters of the CUDA-core kernel show it issue-bound).
//
// Work split is the CUDA-core kernel's (one CTA of 4 warps per work item,
// each warp streams whole 16-token blocks through its own ring of shared
// memory stages filled by 2-D TMA, or by 1-D bulk copies where a row is not
// a multiple of 128 bytes).  Per block a warp computes
//   S^T [16 tokens x 8 heads] = K [16 x D] . Q^T [D x 8]      (M = tokens)
//   O^T [D x 8 heads]        += V^T [D x 16] . P^T [16 x 8]   (M = head dim)
// with G <= 8 query heads in the N = 8 columns.  Operand fragments are
// built straight from the quantised codes in shared memory, dequantised in
// registers to f16 (exact for all three formats: int8 codes, e2m1 * e4m3
// products with at most 6 significant bits, and E4M3 values, whose range
// 2^-9 .. 448 and 4 significant bits f16 holds).  Because a dot product does
// not care in which order it visits the head dim, each lane reads 16
// contiguous bytes of a key row and the query fragments use the same
// permuted head-dim order; for PV the head-dim rows are permuted the same
// way and un-permuted when the output is written.  The scores' fragment
// layout is turned into PV's B fragment by one movmatrix transpose per 8
// tokens.  bf16 KV skips the dequant: K and V^T fragments come from the
// swizzled tiles by ldmatrix (.trans for V, natural head-dim order), q is
// used as bf16 and P enters PV as a bf16 hi + lo pair.
// Scales: int8 per-token scales multiply the score (K) and the
// probability (V); the NVFP4 block scale multiplies the f16 codes (one
// exact f16x2 multiply per pair); softmax_scale * log2 e and the NVFP4 /
// FP8 per-tensor scales are applied in fp32 outside the MMAs, so q stays
// exact.
#pragma once

#include <cuda.h>

#include <cstring>
#include <mutex>

#include "pa_internal.cuh"

namespace pa {
namespace tc {

// ---- 2-D TMA over the pool viewed as [NB * Hkv * 16 token rows, row bytes]
// with 16-row x 128-byte boxes and the 128-byte swizzle: within every 1024
// bytes the 16-byte chunk index of a row is XORed with (row % 8), which makes
// the fragment reads below conflict-free.

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// rows of `row_bytes` (a multiple of 128), boxes of 16 rows x 128 bytes
inline bool make_row_map(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, (cuuint32_t)kBlock};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_rows(void *dst, const CUtensorMap *map, int x, int y,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

// CL: the single-launch variant (one thread-block cluster per sequence and
// kv head, partials merged through distributed shared memory)
template <int DT, int D, bool CL = false>
struct Geo {
  static constexpr bool BF16 = DT == PA_KV_BF16;              // ldmatrix fragments, no dequant
  static constexpr bool BYTE_CODES = DT == PA_KV_INT8 || DT == PA_KV_FP8;   // one byte per element
  static constexpr int ROW = BF16 ? 2 * D : (BYTE_CODES ? D : D / 2);   // bytes per token row
  static constexpr int E = BF16 ? 8 : (BYTE_CODES ? 16 : 32);   // elements per 16 bytes
  static constexpr int KG = D / (4 * E);                      // K chunks per lane
  static constexpr int KS = E / 4;                            // k-steps per K chunk
  // V: the quantised formats read VE elements of 4 tokens per lane chunk; bf16
  // reads 16 x 16 tiles by ldmatrix, one per 16 head-dim rows (VG = D / 16)
  static constexpr int VE = BF16 ? 2 : ((8 * E <= D) ? E : D / 8);
  static constexpr int VB = BYTE_CODES ? VE : VE / 2;        // V chunk bytes (quantised)
  static constexpr int VG = BF16 ? D / 16 : D / (8 * VE);    // V chunk groups
  // scale bytes per token row (FP8 has only the per-tensor scale)
  static constexpr int SROW = DT == PA_KV_INT8 ? 2 : (DT == PA_KV_NVFP4 ? D / 16 : 0);
  static constexpr bool SW = ROW % 128 == 0;                  // TMA tensor copies + swizzle
  static constexpr int CODE = kBlock * ROW;
  static constexpr int SC = kBlock * SROW;
  static constexpr int PAYLOAD = 2 * (CODE + SC);
  static constexpr int STAGE = SW ? (PAYLOAD + 1023) / 1024 * 1024 : PAYLOAD;
  // byte formats: 2 stages so that 3 CTAs (12 warps) fit per SM; NVFP4: 3;
  // bf16 (16 KB per block at D = 256): 1, for 3 CTAs per SM
  // (single-launch variant: 2 stages, so that a warp's first two blocks are
  // in flight together)
  static constexpr int NSTAGE = CL ? 2 : (BF16 ? 1 : (BYTE_CODES ? 2 : 3));
  static constexpr int WARP_BYTES = NSTAGE * STAGE;
  // single-launch variant: the CTA's merged rows [8][D] and their LSE [8],
  // read by the other CTAs of its cluster
  static constexpr int MERGE = CL ? 8 * D * 4 + 8 * 4 : 0;
  static constexpr int SMEM = kWarps * WARP_BYTES + MERGE + (SW ? 1024 : 0);
  static_assert(KG >= 1 && VG >= 1 && CODE % 16 == 0 && SC % 16 == 0, "geometry");
  static_assert(WARP_BYTES >= 8 * D * 4, "stage area holds the warp's O for the merge");
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// four 8x8 matrices of 16-bit elements from shared memory: lanes 8i..8i+7
// give the row addresses of matrix i (16 contiguous bytes each); lane l gets
// row l / 4, elements 2 (l % 4), 2 (l % 4) + 1 of each (.trans: of its transpose)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                        uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &a0, uint32_t &a1,
                                              uint32_t &a2, uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}

// (lo, hi) fp32 -> bf16x2, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// int8 codes -> f16x2, exact: (0x6400 | (code ^ 0x80)) is 1024 + code + 128.
// `x` holds four codes already XORed with 0x80808080; pair 0 = bytes 0,1.
__device__ __forceinline__ uint32_t s8pair_to_h2(uint32_t x, int pair) {
  uint32_t h = prmt(x, 0x64646464u, pair ? 0x4342u : 0x4140u);
  const uint32_t bias = 0x64806480u;   // (1152, 1152) in f16
  __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&h), *reinterpret_cast<const __half2 *>(&bias));
  return *reinterpret_cast<uint32_t *>(&r);
}

// the four bytes (eight E2M1 codes) of a word -> four f16x2, exact; byte j
// -> h[j], low nibble in the low half.  The word is unpacked into byte
// registers once instead of shifting and masking per byte.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// two E4M3 bytes -> f16x2 (lo, hi), exact
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t lo, uint32_t hi) {
  uint32_t r;
  uint16_t pair = (uint16_t)(lo | (hi << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}

// 2^x with the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, which the softmax weights can lose)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// this thread's generic-proxy shared-memory writes -> ordered before later
// async-proxy (bulk copy) writes to the same bytes
__device__ __forceinline__ void fence_async_smem_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// transpose of an 8x8 matrix of 16-bit elements held by the warp (lane i:
// row i / 4, elements 2 (i % 4), 2 (i % 4) + 1)
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// two E4M3 scale bytes (low 16 bits) -> (s0, s0) and (s1, s1) as f16x2
__device__ __forceinline__ void e4m3x2_dup(uint32_t pair, uint32_t &d0, uint32_t &d1) {
  const uint32_t h = e4m3x2_u16_to_h2(pair);
  d0 = prmt(h, h, 0x1010);
  d1 = prmt(h, h, 0x3232);
}

// byte offset of (row, byte) in a tile stored as 16-row x 128-byte boxes
// with the 128-byte swizzle (boxes of 2 KB, one per 128 bytes of row)
__device__ __forceinline__ int sw_off(int row, int byte) {
  return (byte >> 7) * (kBlock * 128) + row * 128 + ((((byte >> 4) & 7) ^ (row & 7)) << 4) +
         (byte & 15);
}

// ---- thread-block clusters (single-launch variant)
constexpr int kMaxCluster = 8;   // CTAs per cluster (the portable limit)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; shared-memory writes before it
// are visible to the cluster's reads after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// a shared-memory address of this CTA -> the same offset in CTA `rank`
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// CL = false: one CTA per planned work item (partials merged by the merge
// kernel).  CL = true: the single-launch variant for small problems -- no
// planner and no merge kernel: cluster i handles (sequence i / Hkv, kv head
// i % Hkv), its CTAs split the sequence's blocks evenly, and after the
// in-CTA merge each CTA merges one slice of the head dim over the cluster's
// partials, read from the other CTAs' shared memory.
template <int DT, int D, int R, bool CL = false>
__global__ void __launch_bounds__(kThreads, 3)
    decode_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using Gm = Geo<DT, D, CL>;
  constexpr int KG = Gm::KG, KS = Gm::KS, VE = Gm::VE, VB = Gm::VB, VG = Gm::VG;
  constexpr int NSTAGE = Gm::NSTAGE, ROW = Gm::ROW, SROW = Gm::SROW;
  constexpr float kRescale = 8.0f;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // swizzled boxes need 1024-byte alignment
  uint8_t *smem = Gm::SW ? smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023) : smem_raw;
  __shared__ __align__(8) uint64_t bars[kWarps][NSTAGE];
  __shared__ float s_m[kWarps][8], s_l[kWarps][8];

  WorkItem it;
  int len;
  if constexpr (CL) {
    // the cluster's (sequence, kv head) and this CTA's share of its blocks
    const int cid = (int)cluster_index(), rank = (int)cluster_rank(), nr = (int)cluster_size();
    const int unit = cid / p.kv.hkv;
    int L = p.seq_lens[unit];
    uint32_t e = 0;
    if (L < 0) {
      e |= PA_ERRF_NEG_LEN;
      L = 0;
    }
    const long long cap = (long long)p.stride * kBlock;
    if (L > cap) {
      e |= PA_ERRF_LEN_OVER_CAPACITY;
      L = (int)cap;
    }
    if (e && rank == 0 && threadIdx.x == 0) set_err(p.hdr, e);
    const int nblk = (L + kBlock - 1) / kBlock, chunk = (nblk + nr - 1) / nr;
    it.unit = unit;
    it.kvh = cid % p.kv.hkv;
    it.blk_begin = min(nblk, rank * chunk);
    it.blk_end = min(nblk, it.blk_begin + chunk);
    it.part = rank;
    it.parts = nr;
    it.slot = -1;
    it.pad = 0;
    len = L;
  } else {
    griddep_launch();   // the merge may start launching once every CTA has begun
    griddep_wait();     // the plan of this call is complete
    const uint32_t num_items = p.hdr[HDR_NUM_ITEMS];
    if (blockIdx.x >= num_items) return;
    it = p.items[blockIdx.x];
    len = p.units[it.unit].len;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int Q = p.Q;
  const int b = p.virt ? it.unit / Q : it.unit;
  const int qi = p.virt ? it.unit % Q : 0;
  const int kvh = it.kvh;
  const int Hkv = p.kv.hkv;

  // ---- query fragments (B operand of S^T = K Q^T), head-dim order permuted
  // like the key fragments: k-step (g, s), rows 2c..2c+1 <-> d = g*4E + c*E + 4s
  // + {0,1}, rows 2c+8.. <-> + {2,3}.  Column n = r is query head r.
  uint32_t qf[KG][KS][2];
  {
    const bool live = r < R;
    const __nv_bfloat16 *qrow =
        p.q + (((size_t)b * Q + qi) * p.Hq + (size_t)kvh * p.G + (live ? r : 0)) * D;
    if constexpr (Gm::BF16) {
      // bf16 keys come by ldmatrix in natural head-dim order: k-step t covers
      // d = 16t .. 16t + 15, rows 2c, 2c+1 <-> d = 16t + 2c + {0,1}, rows
      // 2c+8, 2c+9 <-> + 8; q stays bf16 (exact)
#pragma unroll
      for (int t = 0; t < D / 16; ++t) {
        const int d = 16 * t + 2 * c;
        qf[t / KS][t % KS][0] = live ? *reinterpret_cast<const uint32_t *>(qrow + d) : 0u;
        qf[t / KS][t % KS][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + d + 8) : 0u;
      }
    } else {
#pragma unroll
      for (int g = 0; g < KG; ++g)
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int d = g * 4 * Gm::E + c * Gm::E + 4 * s;
          uint2 u = live ? *reinterpret_cast<const uint2 *>(qrow + d) : make_uint2(0, 0);
          float2 x0 = bf16x2_to_f2(u.x), x1 = bf16x2_to_f2(u.y);
          qf[g][s][0] = f2_to_h2(x0.x, x0.y);
          qf[g][s][1] = f2_to_h2(x1.x, x1.y);
        }
    }
  }
  const float qscale = p.scale_log2 * (has_global_scale(DT) ? p.kv.kg : 1.0f);

  // ---- this warp's blocks
  const int t_begin = it.blk_begin * kBlock;
  const int t_end = min(len, it.blk_end * kBlock);
  const int n_blk = t_end > t_begin ? (t_end - t_begin + kBlock - 1) / kBlock : 0;
  const int n_local = n_blk > warp ? (n_blk - warp + kWarps - 1) / kWarps : 0;

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
  uint32_t valid_bits = 0;
  bool failed = false;
  // test mode (PA_TEST_EXPIRE_WAIT): the copy of each warp's first block is
  // never issued, so the wait for it runs out after kTestWaitCap polls
  const bool withhold = p.test_expire != 0;
  const uint32_t wait_cap = withhold ? kTestWaitCap : kWaitCap;

  auto issue = [&](int j) {
    if (withhold && j == 0) {   // warp-uniform: nothing issued, nothing arrives
      valid_bits &= ~1u;
      return;
    }
    const int chunk = j >> 5;
    if (chunk != tab_chunk) {
      const int jj = chunk * 32 + lane;
      tab_cache = (jj < n_local) ? __ldg(trow + it.blk_begin + warp + jj * kWarps) : -1;
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
        mbar_arrive_expect_tx(bar, Gm::PAYLOAD);
        if constexpr (Gm::SW) {
          const int y = (int)(tile * kBlock);
#pragma unroll
          for (int x = 0; x < ROW; x += 128) {
            tma_rows(st + x * kBlock, &tmK, x, y, bar, pol);
            tma_rows(st + Gm::CODE + x * kBlock, &tmV, x, y, bar, pol);
          }
        } else {
          bulk_g2s(st, (const uint8_t *)p.kv.k + tile * Gm::CODE, Gm::CODE, bar, pol);
          bulk_g2s(st + Gm::CODE, (const uint8_t *)p.kv.v + tile * Gm::CODE, Gm::CODE, bar, pol);
        }
        if constexpr (Gm::SC > 0) {
          bulk_g2s(st + 2 * Gm::CODE, (const uint8_t *)p.kv.ks + tile * Gm::SC, Gm::SC, bar, pol);
          bulk_g2s(st + 2 * Gm::CODE + Gm::SC, (const uint8_t *)p.kv.vs + tile * Gm::SC, Gm::SC,
                   bar, pol);
        }
      }
    }
  };

  // ---- state: columns 2c, 2c+1 (query heads) of this lane
  float m_run[2] = {kNegInf, kNegInf};
  float l_run[2] = {0.f, 0.f};
  float o[VG][VE / 2][4];
#pragma unroll
  for (int g = 0; g < VG; ++g)
#pragma unroll
    for (int e = 0; e < VE / 2; ++e)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[g][e][k] = 0.f;

  const int prologue = min(NSTAGE, n_local);
  for (int j = 0; j < prologue; ++j) issue(j);
  int issued = prologue;

  for (int j = 0; j < n_local; ++j) {
    const int s = j % NSTAGE;
    const bool arrived = mbar_wait(&bars[warp][s], (j / NSTAGE) & 1, wait_cap);
    if (!__all_sync(0xffffffffu, arrived)) {
      failed = true;
      if (lane == 0) set_err(p.hdr, PA_ERRF_WAIT_TIMEOUT);
      break;
    }
    if (valid_bits & (1u << s)) {
      const uint8_t *st = wsm + s * Gm::STAGE;
      const uint8_t *sK = st, *sV = st + Gm::CODE;
      const uint8_t *sKs = st + 2 * Gm::CODE, *sVs = sKs + Gm::SC;
      const int tok0 = t_begin + (warp + j * kWarps) * kBlock;
      const int nvalid = min(kBlock, t_end - tok0);

      // ---- S^T = K . Q^T; int8 alternates k-steps over two accumulators and
      // NVFP4 over four, so that the MMAs form independent dependency chains
      // (FP8 keeps one: it is at its register bound for 3 CTAs per SM)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
      float sacc3[4] = {0.f, 0.f, 0.f, 0.f}, sacc4[4] = {0.f, 0.f, 0.f, 0.f};   // NVFP4, bf16: 4 chains
      if constexpr (Gm::BF16) {
        // k-step t: matrices (tokens 0-7 | 8-15) x (d 16t .. +7 | 16t+8 .. +15);
        // lane l addresses token row (l & 7) + 8 ((l >> 3) & 1), chunk l >> 4
        const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lhalf = lane >> 4;
        const uint32_t kbase = smem_u32(sK);
#pragma unroll
        for (int t = 0; t < D / 16; ++t) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kbase + sw_off(lrow, 32 * t + 16 * lhalf), a0, a1, a2, a3);
          float(&acc)[4] = (t & 3) == 0 ? sacc : (t & 3) == 1 ? sacc2 : (t & 3) == 2 ? sacc3 : sacc4;
          mma16816_bf16(acc, a0, a1, a2, a3, qf[t / KS][t % KS][0], qf[t / KS][t % KS][1]);
        }
      } else {
#pragma unroll
      for (int g = 0; g < KG; ++g) {
        const int boff = g * 64 + c * 16;
        const int koff = Gm::SW ? sw_off(r, boff) : r * ROW + boff;   // row r + 8: same swizzle
        uint4 k0 = *reinterpret_cast<const uint4 *>(sK + koff);
        uint4 k1 = *reinterpret_cast<const uint4 *>(sK + koff + 8 * (Gm::SW ? 128 : ROW));
        uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w1[4] = {k1.x, k1.y, k1.z, k1.w};
        if constexpr (DT == PA_KV_INT8) {
#pragma unroll
          for (int s2 = 0; s2 < KS; ++s2) {   // k-step s2 uses word s2 of each row
            const uint32_t x0 = w0[s2] ^ 0x80808080u, x1 = w1[s2] ^ 0x80808080u;
            mma16816((s2 & 1) ? sacc2 : sacc, s8pair_to_h2(x0, 0), s8pair_to_h2(x1, 0),
                     s8pair_to_h2(x0, 1), s8pair_to_h2(x1, 1), qf[g][s2][0], qf[g][s2][1]);
          }
        } else if constexpr (DT == PA_KV_FP8) {
#pragma unroll
          for (int s2 = 0; s2 < KS; ++s2)   // bytes 0,1 of word s2 -> k rows 2c, 2c+1
            mma16816(sacc, e4m3x2_u16_to_h2(w0[s2]), e4m3x2_u16_to_h2(w1[s2]),
                     e4m3x2_u16_to_h2(w0[s2] >> 16), e4m3x2_u16_to_h2(w1[s2] >> 16),
                     qf[g][s2][0], qf[g][s2][1]);
        } else {
          // the lane's two 16-element scale blocks sb, sb + 1 (sb even): one
          // 16-bit load per row
          const int sb = (g * 4 * Gm::E + c * Gm::E) / 16;
          uint32_t sc00, sc01, sc10, sc11;
          e4m3x2_dup(*reinterpret_cast<const uint16_t *>(sKs + r * SROW + sb), sc00, sc01);
          e4m3x2_dup(*reinterpret_cast<const uint16_t *>(sKs + (r + 8) * SROW + sb), sc10, sc11);
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {   // word wi = k-steps 2 wi, 2 wi + 1
            uint32_t h0[4], h1[4];
            e2m1x8_to_h2x4(w0[wi], h0);
            e2m1x8_to_h2x4(w1[wi], h1);
            const uint32_t a_s = wi < 2 ? sc00 : sc01, b_s = wi < 2 ? sc10 : sc11;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)   // k-step 2 wi + hh = bytes 2 hh, 2 hh + 1
              mma16816((wi & 1) ? (hh ? sacc4 : sacc3) : (hh ? sacc2 : sacc),
                       hmul2_u32(h0[2 * hh], a_s), hmul2_u32(h1[2 * hh], b_s),
                       hmul2_u32(h0[2 * hh + 1], a_s), hmul2_u32(h1[2 * hh + 1], b_s),
                       qf[g][2 * wi + hh][0], qf[g][2 * wi + hh][1]);
          }
        }
      }
      }
      if constexpr (DT == PA_KV_NVFP4 || Gm::BF16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) sacc[k] = (sacc[k] + sacc2[k]) + (sacc3[k] + sacc4[k]);
      } else if constexpr (DT == PA_KV_INT8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) sacc[k] += sacc2[k];
      }
      // scale, mask
      float f0 = qscale, f1 = qscale;
      if constexpr (DT == PA_KV_INT8) {
        f0 *= fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sKs)[r]);
        f1 *= fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sKs)[r + 8]);
      }
      const bool v0 = r < nvalid, v1 = r + 8 < nvalid;
      float sc[4];
      sc[0] = v0 ? sacc[0] * f0 : kNegInf;
      sc[1] = v0 ? sacc[1] * f0 : kNegInf;
      sc[2] = v1 ? sacc[2] * f1 : kNegInf;
      sc[3] = v1 ? sacc[3] * f1 : kNegInf;

      // ---- online softmax over the block's tokens, per column.  The lane's
      // own scores decide whether the running max must move (some score above
      // it by more than kRescale); only then is the column max reduced over
      // the 8 lanes that hold the column.
      float mx[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
      const bool need = (mx[0] > m_run[0] + kRescale) || (mx[1] > m_run[1] + kRescale);
      if (__any_sync(0xffffffffu, need)) {
        float al[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mn = fmaxf(m_run[h], mx[h]);
          al[h] = (mn == kNegInf) ? 1.f : ex2f(m_run[h] - mn);
          m_run[h] = mn;
          l_run[h] *= al[h];
        }
#pragma unroll
        for (int g = 0; g < VG; ++g)
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            o[g][e][0] *= al[0];
            o[g][e][1] *= al[1];
            o[g][e][2] *= al[0];
            o[g][e][3] *= al[1];
          }
      }
      float pr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) pr[k] = (sc[k] == kNegInf) ? 0.f : ex2f(sc[k] - m_run[k & 1]);
      l_run[0] += pr[0] + pr[2];
      l_run[1] += pr[1] + pr[3];
      if constexpr (DT == PA_KV_INT8) {
        const float vs0 = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sVs)[r]);
        const float vs1 = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(sVs)[r + 8]);
        pr[0] = v0 ? pr[0] * vs0 : 0.f;
        pr[1] = v0 ? pr[1] * vs0 : 0.f;
        pr[2] = v1 ? pr[2] * vs1 : 0.f;
        pr[3] = v1 ? pr[3] * vs1 : 0.f;
      }
      // ---- P^T fragment (tokens 2c, 2c+1 | 2c+8, 2c+9; column r): the lane
      // holds P[token r | r + 8][heads 2c, 2c+1], which is the row layout of
      // an 8x8 b16 matrix, so one warp transpose per 8 tokens gives it
      if constexpr (Gm::BF16) {
        // bf16 P as hi + lo (hi = RN(p), lo = RN(p - hi)): about 16 significant
        // bits of each probability reach the PV product
        const uint32_t h0 = f2_to_bf2(pr[0], pr[1]), h1 = f2_to_bf2(pr[2], pr[3]);
        const uint32_t l0 = f2_to_bf2(pr[0] - __uint_as_float(h0 << 16),
                                      pr[1] - __uint_as_float(h0 & 0xffff0000u));
        const uint32_t l1 = f2_to_bf2(pr[2] - __uint_as_float(h1 << 16),
                                      pr[3] - __uint_as_float(h1 & 0xffff0000u));
        const uint32_t B0h = movm_trans(h0), B1h = movm_trans(h1);
        const uint32_t B0l = movm_trans(l0), B1l = movm_trans(l1);
        // rows past the sequence end may hold anything (NaN included): zero
        // them in this warp's own stage so that 0 * garbage never reaches O
        if (nvalid < kBlock) {
          uint8_t *vz = const_cast<uint8_t *>(sV);
          constexpr int RC = ROW / 16;   // 16-byte chunks per row
          for (int i = lane; i < (kBlock - nvalid) * RC; i += 32) {
            const int t = nvalid + i / RC, j = i % RC;
            *reinterpret_cast<uint4 *>(vz + (j >> 3) * (kBlock * 128) + t * 128 + (j & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_async_smem_cta();   // ordered before the next copy into this stage
          __syncwarp();
        }
        // m-tile m: matrices (tokens 0-7 | 8-15) x (d 16m .. +7 | 16m+8 .. +15),
        // transposed: lane l addresses token row (l & 7) + 8 ((l >> 4) & 1),
        // chunk (l >> 3) & 1
        const int vrow = (lane & 7) + ((lane >> 4) & 1) * 8, vhalf = (lane >> 3) & 1;
        const uint32_t vbase = smem_u32(sV);
#pragma unroll
        for (int m = 0; m < VG; ++m) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(vbase + sw_off(vrow, 32 * m + 16 * vhalf), a0, a1, a2, a3);
          mma16816_bf16(o[m][0], a0, a1, a2, a3, B0h, B1h);
          mma16816_bf16(o[m][0], a0, a1, a2, a3, B0l, B1l);
        }
      } else {
      const uint32_t B0 = movm_trans(f2_to_h2(pr[0], pr[1]));
      const uint32_t B1 = movm_trans(f2_to_h2(pr[2], pr[3]));

      // ---- O^T += V^T . P^T ; this lane's tokens 2c, 2c+1, 2c+8, 2c+9
      const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
      for (int g = 0; g < VG; ++g) {
        const int boff = g * 8 * VB + r * VB;
        uint32_t vw[4][VB / 4];
        uint32_t vsb[4][2];   // NVFP4: raw E4M3 scale bytes of the lane's 1-2 blocks
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool ok = tk[t] < nvalid;   // poisoned tail slots must not reach the MMA
          const uint8_t *src = sV + (Gm::SW ? sw_off(tk[t], boff) : tk[t] * ROW + boff);
          if constexpr (VB == 16) {
            uint4 u = ok ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0, 0, 0, 0);
            vw[t][0] = u.x;
            vw[t][1] = u.y;
            vw[t][2] = u.z;
            vw[t][3] = u.w;
          } else {
            uint2 u = ok ? *reinterpret_cast<const uint2 *>(src) : make_uint2(0, 0);
            vw[t][0] = u.x;
            vw[t][1] = u.y;
          }
          if constexpr (DT == PA_KV_NVFP4) {
            const int sb = (g * 8 * VE + r * VE) / 16;
            if constexpr (VE > 16) {   // blocks sb, sb + 1 (sb even): one 16-bit load
              vsb[t][0] = ok ? *reinterpret_cast<const uint16_t *>(sVs + tk[t] * SROW + sb) : 0u;
            } else {
              vsb[t][0] = ok ? sVs[tk[t] * SROW + sb] : 0u;
              vsb[t][0] |= vsb[t][0] << 8;
            }
            vsb[t][1] = 0u;
          } else if constexpr (DT == PA_KV_INT8) {
#pragma unroll
            for (int q = 0; q < VB / 4; ++q) vw[t][q] ^= 0x80808080u;   // offset-binary
            (void)vsb;
          } else {
            (void)vsb;
          }
        }
        if constexpr (DT == PA_KV_NVFP4) {
          // Token pairs (2c, 2c+1) and (2c+8, 2c+9): interleave their nibbles so
          // that byte e of X holds (token a, token b) at head-dim row r and
          // byte e of Y the same at row r + 8 -- each cvt then yields an A
          // register directly.
          // scale pair (token a, token b) of block k: byte k of each token's pair
          uint32_t sp[2][2];
#pragma unroll
          for (int pr2 = 0; pr2 < 2; ++pr2)
#pragma unroll
            for (int k = 0; k < 2; ++k)
              sp[pr2][k] = e4m3x2_u16_to_h2(prmt(vsb[2 * pr2][0], vsb[2 * pr2 + 1][0], k ? 0x51u : 0x40u));
#pragma unroll
          for (int wq = 0; wq < VB / 4; ++wq) {
            uint32_t xa[4], ya[4], xb[4], yb[4];
            e2m1x8_to_h2x4((vw[0][wq] & 0x0F0F0F0Fu) | ((vw[1][wq] << 4) & 0xF0F0F0F0u), xa);
            e2m1x8_to_h2x4(((vw[0][wq] >> 4) & 0x0F0F0F0Fu) | (vw[1][wq] & 0xF0F0F0F0u), ya);
            e2m1x8_to_h2x4((vw[2][wq] & 0x0F0F0F0Fu) | ((vw[3][wq] << 4) & 0xF0F0F0F0u), xb);
            e2m1x8_to_h2x4(((vw[2][wq] >> 4) & 0x0F0F0F0Fu) | (vw[3][wq] & 0xF0F0F0F0u), yb);
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) {
              const int e = wq * 4 + j2;
              const int k = e >= 8 ? 1 : 0;
              mma16816(o[g][e], hmul2_u32(xa[j2], sp[0][k]), hmul2_u32(ya[j2], sp[0][k]),
                       hmul2_u32(xb[j2], sp[1][k]), hmul2_u32(yb[j2], sp[1][k]), B0, B1);
            }
          }
        } else if constexpr (DT == PA_KV_FP8) {
          // Interleave the bytes of token pairs (2c, 2c+1) and (2c+8, 2c+9) so
          // that each 16-bit half is (token a, token b) at one head-dim row:
          // one cvt per A register.  Element pair e = bytes 2(e%2), 2(e%2)+1
          // of word e/2.
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            const uint32_t sel = (e & 1) ? 0x7362u : 0x5140u;
            const uint32_t xa = prmt(vw[0][e >> 1], vw[1][e >> 1], sel);
            const uint32_t xb = prmt(vw[2][e >> 1], vw[3][e >> 1], sel);
            mma16816(o[g][e], e4m3x2_u16_to_h2(xa), e4m3x2_u16_to_h2(xa >> 16),
                     e4m3x2_u16_to_h2(xb), e4m3x2_u16_to_h2(xb >> 16), B0, B1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            uint32_t h[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) h[t] = s8pair_to_h2(vw[t][e >> 1], e & 1);   // zeroed slot -> 0
            mma16816(o[g][e], prmt(h[0], h[1], 0x5410), prmt(h[0], h[1], 0x7632),
                     prmt(h[2], h[3], 0x5410), prmt(h[2], h[3], 0x7632), B0, B1);
          }
        }
      }
      }
    }
    __syncwarp();
    if (issued < n_local) {
      issue(issued);
      ++issued;
    }
  }
  if (failed) {
    // let every copy this warp issued land before the CTA exits.  Only the
    // last fill of each stage can still be in flight (a stage is refilled
    // after its previous fill was consumed), and only its phase may be
    // waited on: an older phase's parity repeats and would read as pending.
    for (int j = max(issued - NSTAGE, withhold ? 1 : 0); j < issued; ++j)
      (void)mbar_wait(&bars[warp][j % NSTAGE], (j / NSTAGE) & 1);
  }

  // ---- per-warp totals
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
  }
  if (r == 0) {
    s_m[warp][2 * c] = m_run[0];
    s_m[warp][2 * c + 1] = m_run[1];
    s_l[warp][2 * c] = l_run[0];
    s_l[warp][2 * c + 1] = l_run[1];
  }
  float *ow = reinterpret_cast<float *>(wsm);   // [8 heads][D]
  if constexpr (Gm::BF16) {   // m-tile g: rows d = 16 g + r and + 8 (natural order)
#pragma unroll
    for (int g = 0; g < VG; ++g) {
      const int d = 16 * g + r;
      ow[(2 * c) * D + d] = o[g][0][0];
      ow[(2 * c + 1) * D + d] = o[g][0][1];
      ow[(2 * c) * D + d + 8] = o[g][0][2];
      ow[(2 * c + 1) * D + d + 8] = o[g][0][3];
    }
  } else {
#pragma unroll
    for (int g = 0; g < VG; ++g)
#pragma unroll
      for (int e = 0; e < VE / 2; ++e) {
        const int d = g * 8 * VE + r * VE + 2 * e;
        *reinterpret_cast<float2 *>(ow + (2 * c) * D + d) = make_float2(o[g][e][0], o[g][e][2]);
        *reinterpret_cast<float2 *>(ow + (2 * c + 1) * D + d) = make_float2(o[g][e][1], o[g][e][3]);
      }
  }
  __syncthreads();

  // ---- merge the warps and write (rows h < R)
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
      const float mw = s_m[w][h];
      const float f = (mw == kNegInf) ? 0.f : exp2f(mw - M);
      L += f * s_l[w][h];
      acc += f * reinterpret_cast<const float *>(smem + w * Gm::WARP_BYTES)[h * D + d];
    }
    const float out = L > 0.f ? acc / L * vg : 0.f;
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : kNegInf;
    if constexpr (CL) {   // this CTA's partial, for the cluster merge below
      float *mo = reinterpret_cast<float *>(smem + kWarps * Gm::WARP_BYTES);
      mo[h * D + d] = out;
      if (d == 0) mo[8 * D + h] = lse;
    } else if (it.parts <= 1) {
      const size_t row = ((size_t)b * Q + qi) * p.Hq + (size_t)kvh * G + h;
      if (p.out_fp32)
        reinterpret_cast<float *>(p.out)[row * D + d] = out;
      else
        reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(out);
      if (d == 0 && p.lse_out) p.lse_out[row] = lse;
    } else {
      const size_t prow = ((size_t)it.slot * Hkv + kvh) * p.R + h;
      p.part_o[prow * D + d] = out;
      if (d == 0) p.part_lse[prow] = lse;
    }
  }
  if constexpr (CL) {
    // LSE merge of the cluster's partials: this CTA takes head-dim slice
    // [d0, d1) of every row
    cluster_sync_all();
    const int rank = (int)cluster_rank(), nr = (int)cluster_size();
    const int per = (D + nr - 1) / nr, d0 = rank * per, d1 = min(D, d0 + per);
    const uint32_t mo = smem_u32(smem + kWarps * Gm::WARP_BYTES);
    for (int idx = threadIdx.x; idx < R * per; idx += kThreads) {
      const int h = idx / per, d = d0 + idx % per;
      if (d >= d1) continue;
      // all 2 * nr remote loads are issued before any result is used (an
      // empty partial holds o = 0 and lse = -inf, both defined)
      float lj[kMaxCluster], oj[kMaxCluster];
#pragma unroll
      for (int j = 0; j < kMaxCluster; ++j) {
        if (j < nr) {
          lj[j] = ld_cluster_f32(map_rank(mo + (uint32_t)(8 * D + h) * 4, (uint32_t)j));
          oj[j] = ld_cluster_f32(map_rank(mo + (uint32_t)(h * D + d) * 4, (uint32_t)j));
        }
      }
      float M = kNegInf;
#pragma unroll
      for (int j = 0; j < kMaxCluster; ++j)
        if (j < nr) M = fmaxf(M, lj[j]);
      float acc = 0.f, wsum = 0.f;
      if (M != kNegInf) {
#pragma unroll
        for (int j = 0; j < kMaxCluster; ++j) {
          if (j < nr) {
            const float w = lj[j] == kNegInf ? 0.f : __expf(lj[j] - M);
            acc += w * oj[j];
            wsum += w;
          }
        }
      }
      const float out = wsum > 0.f ? acc / wsum : 0.f;
      const size_t row = ((size_t)b * Q + qi) * p.Hq + (size_t)kvh * G + h;
      if (p.out_fp32)
        reinterpret_cast<float *>(p.out)[row * D + d] = out;
      else
        reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(out);
      if (d == 0 && p.lse_out) p.lse_out[row] = wsum > 0.f ? M + __logf(wsum) : kNegInf;
    }
    cluster_sync_all();   // no CTA leaves while another still reads its partial
  }
}

template <int DT, int D, int R>
cudaError_t launch_one(const AttnParams &p, int grid, cudaStream_t s) {
  using Gm = Geo<DT, D>;
  auto kern = decode_kernel<DT, D, R>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof tk);
  std::memset(&tv, 0, sizeof tv);
  if constexpr (Gm::SW) {
    const uint64_t rows = (uint64_t)p.kv.num_blocks * p.kv.hkv * kBlock;
    if (!make_row_map(&tk, p.kv.k, Gm::ROW, rows) || !make_row_map(&tv, p.kv.v, Gm::ROW, rows))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, kThreads, Gm::SMEM, s, p, tk, tv);
}

// single-launch variant: B * Hkv clusters of P <= kMaxCluster CTAs
template <int DT, int D, int R>
cudaError_t launch_cluster_one(const AttnParams &p, int P, cudaStream_t s) {
  using Gm = Geo<DT, D, true>;
  auto kern = decode_kernel<DT, D, R, true>;
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof tk);
  std::memset(&tv, 0, sizeof tv);
  if constexpr (Gm::SW) {
    const uint64_t rows = (uint64_t)p.kv.num_blocks * p.kv.hkv * kBlock;
    if (!make_row_map(&tk, p.kv.k, Gm::ROW, rows) || !make_row_map(&tv, p.kv.v, Gm::ROW, rows))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.B * p.kv.hkv * P;
  if (P < 1 || P > kMaxCluster || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

template <int DT>
cudaError_t launch_cluster_dtype(const AttnParams &p, int P, cudaStream_t s) {
  const int D = p.kv.D, R = p.R;
#define PA_TC_CASE(DD, RR) \
  if (D == DD && R == RR) return launch_cluster_one<DT, DD, RR>(p, P, s);
  PA_TC_CASE(128, 1) PA_TC_CASE(128, 2) PA_TC_CASE(128, 4) PA_TC_CASE(128, 6)
  PA_TC_CASE(128, 8) PA_TC_CASE(256, 1) PA_TC_CASE(256, 2) PA_TC_CASE(256, 4)
  PA_TC_CASE(256, 6) PA_TC_CASE(256, 8)
#undef PA_TC_CASE
  return cudaErrorInvalidValue;
}

// CTAs of decode_kernel<DT, D, R> one SM holds at once (0 if unknown)
template <int DT, int D, int R>
int occupancy_one() {
  using Gm = Geo<DT, D>;
  auto kern = decode_kernel<DT, D, R>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, Gm::SMEM) != cudaSuccess)
    return 0;
  return n;
}

template <int DT>
int occupancy_dtype(int D, int R) {
#define PA_TC_CASE(DD, RR) \
  if (D == DD && R == RR) return occupancy_one<DT, DD, RR>();
  PA_TC_CASE(128, 1) PA_TC_CASE(128, 2) PA_TC_CASE(128, 4) PA_TC_CASE(128, 6)
  PA_TC_CASE(128, 8) PA_TC_CASE(256, 1) PA_TC_CASE(256, 2) PA_TC_CASE(256, 4)
  PA_TC_CASE(256, 6) PA_TC_CASE(256, 8)
#undef PA_TC_CASE
  return 0;
}

template <int DT>
cudaError_t launch_dtype(const AttnParams &p, int grid, cudaStream_t s) {
  const int D = p.kv.D, R = p.R;
#define PA_TC_CASE(DD, RR) \
  if (D == DD && R == RR) return launch_one<DT, DD, RR>(p, grid, s);
  PA_TC_CASE(128, 1) PA_TC_CASE(128, 2) PA_TC_CASE(128, 4) PA_TC_CASE(128, 6)
  PA_TC_CASE(128, 8) PA_TC_CASE(256, 1) PA_TC_CASE(256, 2) PA_TC_CASE(256, 4)
  PA_TC_CASE(256, 6) PA_TC_CASE(256, 8)
#undef PA_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tc
}  // namespace pa
