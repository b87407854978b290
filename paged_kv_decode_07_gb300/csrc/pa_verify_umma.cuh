// pa_verify_umma.cuh -- speculative verify on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory) for the NVFP4 and
// FP8-E4M3 KV formats, head dim 256.
//
// The q_len x G query rows of one kv head share every key block ("vLLM
// All-NVFP4 DFlash2 for Blackwell", "What makes this stack different":
// DFlash2 K=7 gives 8 query tokens per verify step; causal among the new
// tokens as in the virtual batch of "vLLM-SM70", "Why": query i sees keys
// t < L - Q + 1 + i).  Per 128-token tile of a work item:
//
//   S^T [128 tokens x N rows] = K [128 x 256] . Q^T [256 x N]
//       A = K, dequantised to f16 straight into tensor memory (one token row
//           per TMEM lane), B = Q (f16, shared memory, K-major, 128-byte
//           swizzle), D = S^T in tensor memory (fp32)
//   O^T [256 x N] += V^T [256 x 16 tokens] . P^T [16 tokens x N], per block
//       A = V^T (f16 in shared memory, MN-major: V rows as written by the
//           dequant), B = P^T (f16, shared memory, K-major over tokens),
//           D = O^T in tensor memory (two 128-lane halves of the head dim)
//
// N = the row group (16, 32 or 48 rows).  With tokens on the MMA's M side
// the whole 48-row group is one instruction wide (N = 48) and nothing is
// padded; at N = 48 an A operand read from shared memory would need more
// shared-memory bandwidth than the MMA's own rate, which is why K goes
// through tensor memory.
//
// One persistent CTA per SM walks its work items (the planner's split-K
// partitions) with warp-specialised roles:
//   warps 0, 3   producers (K side, V side): TMA copies of each 16-token
//                block's codes (and NVFP4 block scales) into rings of raw
//                stages; the two sides sit in different warps so that a
//                wait on one ring never holds back the copies of the other
//   warp 1       tensor-memory allocation; one thread issues the QK MMAs
//   warp 2       one thread issues the PV MMAs (both head-dim halves)
//   warps 4-7    K dequant: token row t of the tile -> TMEM lane t (f16x2)
//   warps 8-15   softmax, two groups of 4 warps, each with half of the N
//                columns: S^T from tensor memory, masks, online softmax in
//                the log2 domain with a lazy rescale (threshold 8), P^T to
//                shared memory; at the end of an item O^T / l to the output
//                or to the split-K partials (merged afterwards)
//   warps 16-19  V dequant: token rows -> the f16 V tile in shared memory
//                (MN-major A operand layout), one half tile (64 tokens) at
//                a time, two threads per row, so that the PV MMAs of one
//                half run while the other half is dequantised
// A warp reaches the tensor-memory lanes 32 (warp % 4) .. + 31, so each
// group of 4 consecutive warps covers all 128 lanes.
// Hand-offs are mbarriers (tcgen05.commit for the MMA side); every wait is
// capped and a timeout sets PA_ERRF_WAIT_TIMEOUT and stops the CTA.
//
// Values: every NVFP4 product e2m1 * e4m3 and every E4M3 value is exact in
// f16; q enters as f16 (exact in f16's normal range); P is rounded to f16
// (p <= 2^8 under the lazy rescale); accumulation is fp32.  softmax_scale,
// log2 e and the per-tensor scales are applied in fp32 outside the MMAs.
#pragma once

#include "pa_decode_mma.cuh"

namespace pa {
namespace umma {

// ------------------------------------------------------------ tcgen05 PTX

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// arrives once on `bar` when every MMA this thread issued so far completes
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// D (tmem) (+)= A (tmem) . B (smem descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// D (tmem) (+)= A (smem descriptor) . B (smem descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane (32x32b shape: warp
// w % 4 reaches lanes 32 (w % 4) .. + 31); the wait is in the same statement
// so no use of the registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15])
      : "r"(taddr)
      : "memory");
}
// 32 / 48 consecutive columns, issued together with one wait
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr), "r"(taddr + 16)
      : "memory");
}
__device__ __forceinline__ void tmem_ld48(uint32_t taddr, float (&v)[48]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31]), "=f"(v[32]), "=f"(v[33]), "=f"(v[34]), "=f"(v[35]), "=f"(v[36]), "=f"(v[37]), "=f"(v[38]), "=f"(v[39]), "=f"(v[40]), "=f"(v[41]), "=f"(v[42]), "=f"(v[43]), "=f"(v[44]), "=f"(v[45]), "=f"(v[46]), "=f"(v[47])
      : "r"(taddr), "r"(taddr + 16), "r"(taddr + 32)
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
      " tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7])
      : "r"(taddr)
      : "memory");
}
// 24 columns as three 8-column loads: every load starts at a multiple of its
// own width (the second softmax group's columns start at 24)
__device__ __forceinline__ void tmem_ld24(uint32_t taddr, float (&v)[24]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23])
      : "r"(taddr), "r"(taddr + 8), "r"(taddr + 16)
      : "memory");
}
// N columns (8, 16, 24, 32 or 48) of this thread's lane
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[N]) {
  static_assert(N == 8 || N == 16 || N == 24 || N == 32 || N == 48, "column count");
  if constexpr (N == 8) tmem_ld8(taddr, v);
  else if constexpr (N == 16) tmem_ld16(taddr, v);
  else if constexpr (N == 24) tmem_ld24(taddr, v);
  else if constexpr (N == 32) tmem_ld32(taddr, v);
  else tmem_ld48(taddr, v);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory accesses by 32-bit address.  Written as PTX so the compiler
// sees no store through a generic pointer that could alias locals (which
// would force every loop-invariant value to be reloaded after each store);
// ordering against barriers comes from the barriers' own memory clobbers.
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ int4 lds_s4(uint32_t a) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w));
}
// 2^x by the MUFU instruction (relative error ~2^-22; results below 2^-126
// flush to zero, far below what a probability can contribute here)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(v));
}

// per-warpgroup register budget (all 4 warps of the group execute it)
template <int R>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
// Moves this warpgroup from the launch count `From` to `To` registers per
// thread: .inc only raises and .dec only lowers the current count (the other
// direction is undefined), so the direction is chosen here, never by hand.
template <int From, int To>
__device__ __forceinline__ void setmaxnreg_to() {
  static_assert(To % 8 == 0 && To >= 24 && To <= 256, "setmaxnreg count");
  if constexpr (To > From) setmaxnreg_inc<To>();
  else if constexpr (To < From) setmaxnreg_dec<To>();
}

// generic-proxy shared-memory writes -> visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// barrier over `n` threads that also ORs a predicate across them
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29), stride byte offset >> 4 (32-45), the constant 1 at
// bit 46, layout 2 = 128-byte swizzle (61-63).  K-major swizzled tiles:
// rows of 128 bytes, 8-row groups `sbo` apart (the leading offset is not
// used).  MN-major swizzled tiles: 64-element MN atoms `lbo` apart, 8-row
// K groups `sbo` apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), A major (bit 15: 0 K, 1 MN), B K-major (bit 16 = 0),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- geometry

constexpr int D = 256;
constexpr int kTile = 128;                 // tokens per QK tile (the MMA's M)
constexpr int kTileBlocks = kTile / kBlock;
constexpr int kThreads = 640;              // 5 warpgroups
constexpr int kLaunchRegs = 96;            // per thread at launch: 65536 / 640, to a multiple of 8
// Registers per thread of each warpgroup after the split: producer/MMA 56,
// K dequant 112, each of the two softmax groups 120, V dequant 72.  Per SM
// sub-partition (one warp of each group) 480 = 5 x 96, so every
// setmaxnreg.inc is satisfied by the decreases.
constexpr int kRegCtl = 56, kRegK = 112, kRegSoftmax = 120, kRegV = 72;
static_assert(kRegCtl + kRegK + 2 * kRegSoftmax + kRegV <= 5 * kLaunchRegs, "register split");
static_assert(kLaunchRegs == 65536 / kThreads / 8 * 8, "launch register count");
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns (32-bit each): two K tiles (128 tokens x 256 f16,
// 128 columns each), two S buffers (64 columns each, N used), one O^T of two
// 128-lane halves (64 columns each, N used)
constexpr uint32_t kColK = 0, kColS = 256, kColO = 384;
// named barriers (0 is __syncthreads)
constexpr uint32_t kBarSoftmax = 1, kBarK = 2, kBarSoftmax1 = 3;

template <int DT, int N>
struct Geo {
  static_assert(DT == PA_KV_NVFP4 || DT == PA_KV_FP8, "NVFP4 and FP8 KV");
  static_assert(N == 16 || N == 32 || N == 48, "row groups of 16, 32 or 48");
  static constexpr int ROW = DT == PA_KV_NVFP4 ? D / 2 : D;     // code bytes per token row
  static constexpr int SROW = DT == PA_KV_NVFP4 ? D / 16 : 0;   // scale bytes per token row
  static constexpr int CODE = kBlock * ROW;
  static constexpr int SC = kBlock * SROW;
  // K and V codes arrive in two rings of raw stages, so that the K side of
  // the next tiles is fetched while the V dequant (which trails by about a
  // tile) still holds its stage.  Raw stage of one tile and side:
  // [codes of 8 blocks][scales of 8 blocks] (every 2 KB code box stays 1 KB
  // aligned for the 128-byte swizzle).
  static constexpr int RSIDE = (kTileBlocks * (CODE + SC) + 1023) / 1024 * 1024;
  static constexpr int R_SC = kTileBlocks * CODE;
  // Ring slots belong to a block's position in its tile: stage
  // (tile % NR) * 8 + j holds block j of a tile, so each stage always has
  // the same consumer threads and no waiter can run two phases ahead of a
  // stage (partial tiles leave stages unused instead of shifting the block
  // -> stage map).  The f16 V of a tile (8 blocks) is handed over as a whole.
  static constexpr int NRK = DT == PA_KV_NVFP4 ? 4 : 2;   // K tiles in flight
  static constexpr int NRV = DT == PA_KV_NVFP4 ? 2 : 1;   // V tiles in flight
  static constexpr int OFF_RK = 0, OFF_RV = NRK * RSIDE;
  static constexpr int VSLOT = kBlock * D * 2;                   // f16 V of one block
  static constexpr int NV = kTileBlocks;
  static constexpr int QCH = N * 128;   // one 64-wide K-major chunk of N rows
  static constexpr int QBUF = 4 * QCH;  // Q: 256 = 4 chunks of 64
  static constexpr int PBUF = 2 * QCH;  // P^T: 128 tokens = 2 chunks of 64
  static constexpr int OFF_V = OFF_RV + NRV * RSIDE;
  static constexpr int OFF_Q = OFF_V + NV * VSLOT;
  static constexpr int OFF_P = OFF_Q + QBUF;
  static constexpr int BYTES = OFF_P + 2 * PBUF;
  static constexpr int SMEM = BYTES + 1024;   // + alignment slack
  static_assert(NRK <= 4 && NRV <= 4, "ring sizes (control block)");
  static_assert(QCH % 1024 == 0 && RSIDE % 1024 == 0 && VSLOT % 1024 == 0 && CODE % 1024 == 0,
                "1 KB atoms");
  static_assert(SMEM + 4096 <= 227 * 1024, "shared memory (with the static control block)");
};

// byte offset of f16 element (row, k) in a K-major tile of 128-byte rows,
// 64-element chunks `chunk` bytes apart, 128-byte swizzle
__device__ __forceinline__ uint32_t kmaj_off(int row, int k, int chunk) {
  return (uint32_t)((k >> 6) * chunk + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                    ((k & 7) << 1));
}


// ------------------------------------------------------------ shared state

constexpr int kMaxN = 48;
constexpr int kMaxNR = 32;

struct Ctl {
  uint64_t rkfull[kMaxNR], rkfree[kMaxNR];     // K raw stages: TMA -> K dequant
  uint64_t rvfull[kMaxNR], rvfree[kMaxNR];     // V raw stages: TMA -> V dequant
  uint64_t vfull[2], vfree[2];                 // f16 V half tiles: V dequant <-> PV
  uint64_t kfull[2], kfree[2];                 // K buffers in tensor memory: K dequant <-> QK
  uint64_t sfull[2], sfree[2];                 // S buffers: QK <-> softmax
  uint64_t pfull[2], pdone[2];                 // P buffers: softmax <-> PV
  uint64_t odone, ofree;                       // O^T: last PV of an item <-> epilogue
  uint64_t done;                               // every MMA of the CTA complete
  uint32_t tmem;                               // tensor-memory base address
  int abort;                                   // a capped wait ran out somewhere
  int rkvalid[kMaxNR], rvvalid[kMaxNR];        // raw stage holds a valid block
  alignas(16) float m[kMaxN];                  // running max of each row (log2 domain)
  alignas(16) float mnew[kMaxN], alpha[kMaxN], inv[kMaxN];
  alignas(16) float red[4][kMaxN];
  alignas(16) int lim[kMaxN];                  // keys visible to each row
  alignas(16) int orow[kMaxN];                 // output (or split-K partial) row of each row
};

// a work item as every role sees it
struct Item {
  WorkItem it;
  int b, ro, kvh, R, L, t_begin, t_end, n_blk, ntiles;
  const int *trow;
};

__device__ __forceinline__ Item load_item(const AttnParams &p, int ii) {
  Item x;
  x.it = p.items[ii];
  x.b = x.it.unit / p.RG;
  x.ro = (x.it.unit % p.RG) * p.R;
  x.kvh = x.it.kvh;
  x.R = min(p.R, p.Q * p.G - x.ro);
  x.L = p.units[x.it.unit].len;
  x.t_begin = x.it.blk_begin * kBlock;
  x.t_end = min(x.L, x.it.blk_end * kBlock);
  x.n_blk = x.t_end > x.t_begin ? (x.t_end - x.t_begin + kBlock - 1) / kBlock : 0;
  x.ntiles = (x.n_blk + kTileBlocks - 1) / kTileBlocks;
  x.trow = p.tables + (size_t)x.b * p.stride;
  return x;
}

// true when the phase with the given parity has completed; a thread whose
// phase is not complete yet sleeps in the hardware (up to `ns` nanoseconds)
// instead of spinning, so waiting warps take no issue slots or shared-memory
// bandwidth from the warps that work
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// non-blocking check of the same phase
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr uint32_t kSleepNs = 20000;        // one suspension: 20 us at most
constexpr uint32_t kSleepCap = 1u << 16;    // => a wait gives up after ~1.3 s

// capped wait that also gives up once another role has given up (the loop
// stays rolled: every call site would otherwise carry unrolled copies, and
// the kernel's code must fit the instruction caches of four roles at once)
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Ctl &c, uint32_t *hdr) {
  if (mbar_test(bar, parity)) return true;   // already complete: no suspension
  volatile int *ab = &c.abort;
#pragma unroll 1
  for (uint32_t i = 0; i < kSleepCap; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if (*ab) return false;
  }
  *ab = 1;
  set_err(hdr, PA_ERRF_WAIT_TIMEOUT);
  return false;
}

// capped wait without the abort check (draining before exit)
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
#pragma unroll 1
  for (uint32_t i = 0; i < kSleepCap; ++i)
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return;
}

// ------------------------------------------------------------------ roles

// warp 0 (K side) or warp 3 (V side): lane j (0-7) copies its side of block
// j of every tile into stage (tile % NRK) * 8 + j (K) or (tile % NRV) * 8 +
// j (V) (code tiles by 2-D TMA with 128-byte swizzle, NVFP4 block scales by
// 1-D bulk copies).  One lane per block position issues a tile's copies in
// parallel and keeps its stage counters and the next tile's block id in
// registers.
template <int DT, int N>
__device__ void role_producer(const AttnParams &p, const CUtensorMap *tmK, const CUtensorMap *tmV,
                              uint8_t *smem, Ctl &c, int num_items, int jt, int side) {
  using Gm = Geo<DT, N>;
  const uint64_t pol = policy_evict_first();
  // this lane's ring: the K or the V side
  const int nr = side ? Gm::NRV : Gm::NRK;
  uint64_t *const full = side ? c.rvfull : c.rkfull;
  uint64_t *const free_ = side ? c.rvfree : c.rkfree;
  int *const rvalid = side ? c.rvvalid : c.rkvalid;
  const CUtensorMap *const tm = side ? tmV : tmK;
  const uint8_t *const scales = static_cast<const uint8_t *>(side ? p.kv.vs : p.kv.ks);
  uint8_t *const base = smem + (side ? Gm::OFF_RV : Gm::OFF_RK);
  uint32_t ruse[4] = {0u, 0u, 0u, 0u};   // fills of this lane's stages so far
  uint32_t g = 0;
  bool ok = true;
  for (int ii = blockIdx.x; ii < num_items && ok; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    // this lane's block id of the next tile is read one tile ahead
    int nxt = jt < x.n_blk ? x.trow[x.it.blk_begin + jt] : -1;
    for (int tile = 0; tile < x.ntiles && ok; ++tile, ++g) {
      const int nb = min(kTileBlocks, x.n_blk - tile * kTileBlocks);
      const int phys = nxt;
      const int j2 = (tile + 1) * kTileBlocks + jt;
      nxt = j2 < x.n_blk ? x.trow[x.it.blk_begin + j2] : -1;
      if (jt >= nb) continue;
      const int stage = (int)(g % (uint32_t)nr);
      const int s = stage * kTileBlocks + jt;
      uint32_t use = 0;
#pragma unroll
      for (int a = 0; a < 4; ++a)
        if (a == stage) use = ruse[a];
      if (!wait_bar(&free_[s], (use & 1) ^ 1, c, p.hdr)) {
        ok = false;
        break;
      }
      // counted once the stage is this lane's to fill: the drain below waits
      // for the phase of the last fill actually issued
#pragma unroll
      for (int a = 0; a < 4; ++a)
        if (a == stage) ++ruse[a];
      const bool v = phys >= 0 && phys < p.kv.num_blocks;
      rvalid[s] = v;
      if (!v) {
        if (side == 0) set_err(p.hdr, PA_ERRF_BAD_BLOCK_ID);
        mbar_arrive(&full[s]);
        continue;
      }
      uint8_t *st = base + stage * Gm::RSIDE;
      const size_t tile_id = (size_t)phys * p.kv.hkv + x.kvh;
      const int y = (int)(tile_id * kBlock);
      mbar_arrive_expect_tx(&full[s], Gm::CODE + Gm::SC);
#pragma unroll
      for (int xo = 0; xo < Gm::ROW; xo += 128)
        tc::tma_rows(st + jt * Gm::CODE + xo * kBlock, tm, xo, y, &full[s], pol);
      if constexpr (Gm::SC > 0)
        bulk_g2s(st + Gm::R_SC + jt * Gm::SC, scales + tile_id * Gm::SC, Gm::SC, &full[s], pol);
    }
  }
  // the last fill of each of this lane's stages may still be in flight after
  // a failure: let the copies land before the CTA exits
#pragma unroll
  for (int a = 0; a < 4; ++a)
    if (ruse[a] > 0) drain_wait(&full[a * kTileBlocks + jt], (ruse[a] - 1) & 1);
}

// Two MMA-issuing threads, each with its own accumulators and commit
// barriers, so that neither stream waits behind the other: QK of tile g
// needs only its K tile and a free S buffer, PV of tile g only its P and V.
// warp 1, one thread: S^T(g) = K(g) . Q^T
template <int DT, int N>
__device__ void role_qk(const AttnParams &p, uint8_t *smem, Ctl &c, uint32_t tmem,
                        int num_items) {
  using Gm = Geo<DT, N>;
  constexpr uint32_t IQK = idesc_f16(kTile, N, false);
  // the descriptor is built once; a k-step moves the start address, which is
  // the low field (address >> 4), by a constant
  const uint64_t dQ = sdesc(smem_u32(smem + Gm::OFF_Q), 16, 1024);
  uint32_t g = 0;
  bool ok = true;
  for (int ii = blockIdx.x; ii < num_items && ok; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    for (int tile = 0; tile < x.ntiles; ++tile, ++g) {
      if (!wait_bar(&c.kfull[g & 1], (g >> 1) & 1, c, p.hdr) ||
          !wait_bar(&c.sfree[g & 1], ((g >> 1) & 1) ^ 1, c, p.hdr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dS = tmem + kColS + (g & 1) * 64;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ts(dS, tmem + kColK + (g & 1) * 128 + ks * 8,
               dQ + (uint64_t)(((ks >> 2) * Gm::QCH + (ks & 3) * 32) >> 4),
               IQK, ks > 0 ? 1u : 0u);
      tc_commit(&c.sfull[g & 1]);
      tc_commit(&c.kfree[g & 1]);
    }
  }
  tc_commit(&c.done);   // tensor memory is released only after every MMA completes
  drain_wait(&c.done, 0);
}

// warp 2, one thread: O^T[half h] += V^T(g)[half h] . P^T(g) per 16-token
// block and head-dim half h (the MMAs of a block run at the tensor pipe's
// rate for shared-memory operands, about 95 cycles each at N <= 48, so one
// issuing thread keeps up).  The V tile arrives in two half tiles of four
// blocks: the MMAs of a half start once its dequant is done, and the half's
// buffer is handed back once they complete.
template <int DT, int N>
__device__ void role_pv(const AttnParams &p, uint8_t *smem, Ctl &c, uint32_t tmem,
                        int num_items) {
  using Gm = Geo<DT, N>;
  constexpr uint32_t IPV = idesc_f16(kTile, N, true);
  const uint32_t sP = smem_u32(smem + Gm::OFF_P);
  const uint64_t dP0 = sdesc(sP, 16, 1024), dP1 = sdesc(sP + Gm::PBUF, 16, 1024);
  // head-dim half 1 starts 4 KB (two 64-wide chunks) into each block's slot
  const uint64_t dV = sdesc(smem_u32(smem + Gm::OFF_V), 2048, 1024);
  constexpr uint64_t kHalf1 = 4096 >> 4;
  const uint32_t dO = tmem + kColO;
  uint32_t g = 0, oi = 0;
  bool ok = true;
  for (int ii = blockIdx.x; ii < num_items && ok; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    if (x.n_blk == 0) continue;
    for (int tile = 0; tile < x.ntiles; ++tile, ++g) {
      const int nb = min(kTileBlocks, x.n_blk - tile * kTileBlocks);
      const bool first = tile == 0;
      if (!wait_bar(&c.pfull[g & 1], (g >> 1) & 1, c, p.hdr) ||
          (first && !wait_bar(&c.ofree, (oi & 1) ^ 1, c, p.hdr))) {
        ok = false;
        break;
      }
      const uint64_t dP = (g & 1) ? dP1 : dP0;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {   // half tiles: blocks 4 hh .. 4 hh + 3
        if (!wait_bar(&c.vfull[hh], g & 1, c, p.hdr)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int j = 4 * hh; j < min(nb, 4 * hh + 4); ++j) {
          const uint64_t bd = dP + (uint64_t)(((j >> 2) * Gm::QCH + (j & 3) * 32) >> 4);
          const uint64_t ad = dV + (uint64_t)((j * Gm::VSLOT) >> 4);
          const uint32_t acc = (first && j == 0) ? 0u : 1u;
          mma_ss(dO, ad, bd, IPV, acc);
          mma_ss(dO + 64, ad + kHalf1, bd, IPV, acc);
        }
        tc_commit(&c.vfree[hh]);
      }
      if (!ok) break;
      tc_commit(&c.pdone[g & 1]);
      if (tile == x.ntiles - 1) tc_commit(&c.odone);
    }
    ++oi;
  }
  tc_commit(&c.done);
  drain_wait(&c.done, 0);
}


// Token row r of a raw stage dequantised to f16, 32 head-dim elements at a
// time (the 64-element pieces u2b .. u2e - 1 of the row, all of it by
// default): sink(u, h) gets h[k] = (element 32u + 2k, element 32u + 2k + 1)
// as f16x2 (low half first).  An invalid row yields zeros (codes and scales
// are not read: poisoned slots may hold NaN scales).  Every lane runs the
// same instruction sequence whether its row is valid or not (zeros are
// selected, not branched to): a K sink is a warp-wide tcgen05.st, which
// all 32 lanes must execute together.
template <int DT, int UU, typename Sink>
__device__ __forceinline__ void deq_row(uint32_t st, int code_off, int scale_off, int r,
                                        bool valid, Sink &&sink, int u2b = 0, int u2e = 4) {
  static_assert(UU == 1 || UU == 2, "chunks in flight");
  const uint4 z = make_uint4(0, 0, 0, 0);
  if constexpr (DT == PA_KV_NVFP4) {
    // chunks 2 u2 and 2 u2 + 1 use the row's scale bytes 4 u2 .. 4 u2 + 3
#pragma unroll 1
    for (int u2 = u2b; u2 < u2e; ++u2) {
      const uint32_t sw = valid ? lds_u32(st + scale_off + r * 16 + 4 * u2) : 0u;
      uint32_t sd[4];
      tc::e4m3x2_dup(sw & 0xffffu, sd[0], sd[1]);
      tc::e4m3x2_dup(sw >> 16, sd[2], sd[3]);
#pragma unroll UU
      for (int uu = 0; uu < 2; ++uu) {
        const int u = 2 * u2 + uu;
        const uint4 w = valid ? lds_u4(st + code_off + tc::sw_off(r, 16 * u)) : z;
        uint32_t h0[4], h1[4], h2[4], h3[4];
        tc::e2m1x8_to_h2x4(w.x, h0);
        tc::e2m1x8_to_h2x4(w.y, h1);
        tc::e2m1x8_to_h2x4(w.z, h2);
        tc::e2m1x8_to_h2x4(w.w, h3);
        const uint32_t s0 = uu ? sd[2] : sd[0], s1 = uu ? sd[3] : sd[1];
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          h[k] = hmul2_u32(h0[k], s0);
          h[4 + k] = hmul2_u32(h1[k], s0);
          h[8 + k] = hmul2_u32(h2[k], s1);
          h[12 + k] = hmul2_u32(h3[k], s1);
        }
        sink(u, h);
      }
    }
  } else {   // FP8-E4M3: one byte per element, exact in f16
#pragma unroll 1
    for (int u = 2 * u2b; u < 2 * u2e; ++u) {
      const uint4 w0 = valid ? lds_u4(st + code_off + tc::sw_off(r, 32 * u)) : z;
      const uint4 w1 = valid ? lds_u4(st + code_off + tc::sw_off(r, 32 * u + 16)) : z;
      const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t h[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        h[2 * k] = e4m3x2_u16_to_h2(wd[k]);
        h[2 * k + 1] = e4m3x2_u16_to_h2(wd[k] >> 16);
      }
      sink(u, h);
    }
  }
}

// Q rows of an item as the QK B operand: f16, K-major, 128-byte swizzle,
// rows >= R zero.  Thread t of the K dequant group loads N / 4 16-byte
// pieces (load_q, issued early so the latency overlaps other work) and
// stores them (store_q).
template <int N>
__device__ __forceinline__ void load_q(const AttnParams &p, const Item &x, int t,
                                       uint4 (&qv)[N / 4]) {
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const int i = t + 128 * k, n = i >> 5, d0 = (i & 31) << 3;
    qv[k] = make_uint4(0, 0, 0, 0);
    if (n < x.R) {
      const int qi = (x.ro + n) / p.G, gg = (x.ro + n) % p.G;
      qv[k] = *reinterpret_cast<const uint4 *>(
          p.q + (((size_t)x.b * p.Q + qi) * p.Hq + (size_t)x.kvh * p.G + gg) * D + d0);
    }
  }
}
template <int N>
__device__ __forceinline__ void store_q(const uint4 (&qv)[N / 4], uint8_t *sQ, int t) {
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const int i = t + 128 * k, n = i >> 5, d0 = (i & 31) << 3;
    const uint4 u = qv[k];
    const float2 a = bf16x2_to_f2(u.x), b = bf16x2_to_f2(u.y), c2 = bf16x2_to_f2(u.z),
                 e = bf16x2_to_f2(u.w);
    sts_u4(smem_u32(sQ) + kmaj_off(n, d0, N * 128), tc::f2_to_h2(a.x, a.y), tc::f2_to_h2(b.x, b.y),
           tc::f2_to_h2(c2.x, c2.y), tc::f2_to_h2(e.x, e.y));
  }
}

// warps 4-7: token row t of each tile -> tensor-memory lane t; at an item's
// first tile also the item's Q (the previous item's QKs are complete then)
template <int DT, int N>
__device__ void role_kdeq(const AttnParams &p, uint8_t *smem, Ctl &c, uint32_t tmem,
                          int num_items, int warp, int lane) {
  using Gm = Geo<DT, N>;
  const int q4 = warp & 3, t = q4 * 32 + lane, jb = t >> 4, r = t & 15;
  const uint32_t ta0 = tmem + ((uint32_t)(q4 * 32) << 16) + kColK;
  uint32_t g = 0, ru[Gm::NRK] = {};   // uses of this row's raw stages
  bool failed = false;
  for (int ii = blockIdx.x; ii < num_items && !failed; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    if (x.n_blk == 0) continue;
    for (int tile = 0; tile < x.ntiles; ++tile) {
      const int nb = min(kTileBlocks, x.n_blk - tile * kTileBlocks);
      const bool have = jb < nb;
      const uint32_t tp = g % Gm::NRK;
      const int s = (int)tp * kTileBlocks + jb;
      uint4 qv[N / 4];
      if (tile == 0) load_q<N>(p, x, t, qv);   // in flight while the previous QK finishes
      uint32_t use = 0;
#pragma unroll
      for (int i = 0; i < Gm::NRK; ++i)
        if (i == (int)tp) use = ru[i];
      // K buffer g % 2 is free once QK(g - 2) completed; the q tile of a new
      // item may be written once QK(g - 1), the last of the previous item, is
      const uint32_t kb = g & 1;
      bool ok = wait_bar(&c.kfree[kb], ((g >> 1) & 1) ^ 1, c, p.hdr);
      if (ok && tile == 0 && g > 0) ok = wait_bar(&c.kfree[kb ^ 1], ((g - 1) >> 1) & 1, c, p.hdr);
      const uint32_t ta = ta0 + kb * 128;
      if (ok && have) ok = wait_bar(&c.rkfull[s], use & 1, c, p.hdr);
      if (named_sync_or(kBarK, 128, !ok)) {   // the whole group stops together
        failed = true;
        break;
      }
      tc_fence_after();
      if (tile == 0) store_q<N>(qv, smem + Gm::OFF_Q, t);
      const int tok = x.t_begin + (tile * kTileBlocks + jb) * kBlock + r;
      const bool valid = have && c.rkvalid[s] != 0 && tok < x.t_end;
      deq_row<DT, 2>(smem_u32(smem) + Gm::OFF_RK + tp * Gm::RSIDE, jb * Gm::CODE, Gm::R_SC + jb * Gm::SC, r, valid,
                  [&](int u, const uint32_t(&h)[16]) { tmem_st16(ta + 16 * u, h); });
      tmem_st_wait();
      if (tile == 0) fence_async_smem();   // Q, written by this thread, for the MMA
      tc_fence_before();
      mbar_arrive(&c.kfull[kb]);
      if (have) {
        mbar_arrive(&c.rkfree[s]);
#pragma unroll
        for (int i = 0; i < Gm::NRK; ++i)
          if (i == (int)tp) ++ru[i];
      }
      ++g;
    }
  }
}

// warps 16-19: the V tile in two half tiles of four blocks; in half hh warp
// w takes block 4 hh + w, lane l row l % 16 and head-dim half l / 16 of it
// -> the block's f16 V slot, laid out [64-wide head-dim chunk][16 tokens]
// [128 bytes, swizzled] (MN-major A of PV)
template <int DT, int N>
__device__ void role_vdeq(const AttnParams &p, uint8_t *smem, Ctl &c, int num_items, int warp,
                          int lane) {
  using Gm = Geo<DT, N>;
  const int w = warp & 3, r = lane & 15, dh = lane >> 4;
  uint32_t g = 0, ru[2][Gm::NRV] = {};   // uses of this thread's raw stages, per half
  bool ok = true;
  for (int ii = blockIdx.x; ii < num_items && ok; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    if (x.n_blk == 0) continue;
    for (int tile = 0; tile < x.ntiles && ok; ++tile, ++g) {
      const int nb = min(kTileBlocks, x.n_blk - tile * kTileBlocks);
      const uint32_t tp = g % Gm::NRV;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int jb = 4 * hh + w;
        // the half's buffer is free once its MMAs of the previous tile completed
        ok = wait_bar(&c.vfree[hh], (g & 1) ^ 1, c, p.hdr);
        if (!ok) break;
        if (jb < nb) {
          const int s = (int)tp * kTileBlocks + jb;
          uint32_t use = 0;
#pragma unroll
          for (int i = 0; i < Gm::NRV; ++i)
            if (i == (int)tp) use = hh ? ru[1][i] : ru[0][i];
          ok = wait_bar(&c.rvfull[s], use & 1, c, p.hdr);
          if (!ok) break;
#pragma unroll
          for (int i = 0; i < Gm::NRV; ++i)
            if (i == (int)tp) {
              if (hh) ++ru[1][i];
              else ++ru[0][i];
            }
          const int tok = x.t_begin + (tile * kTileBlocks + jb) * kBlock + r;
          const bool valid = c.rvvalid[s] != 0 && tok < x.t_end;
          const uint32_t vsl = smem_u32(smem) + Gm::OFF_V + jb * Gm::VSLOT + r * 128;
          deq_row<DT, 2>(smem_u32(smem) + Gm::OFF_RV + tp * Gm::RSIDE, jb * Gm::CODE,
                         Gm::R_SC + jb * Gm::SC, r, valid,
                         [&](int u, const uint32_t(&h)[16]) {
#pragma unroll
                           for (int q = 0; q < 4; ++q)
                             sts_u4(vsl + (u >> 1) * 2048 + (((((u & 1) << 2) + q) ^ (r & 7)) << 4),
                                    h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                         },
                         2 * dh, 2 * dh + 2);
          fence_async_smem();
          mbar_arrive(&c.rvfree[s]);
        }
        mbar_arrive(&c.vfull[hh]);   // every V thread, every half tile
      }
    }
  }
}

// One reduction step over lane bit `bit`: the lane with the bit set keeps
// the upper half of the columns, its partner the lower half.
template <int S, bool MAX>
__device__ __forceinline__ void rs_half(const float (&a)[S], float (&b)[S / 2], int lane, int bit) {
  const bool up = (lane >> bit) & 1;
#pragma unroll
  for (int k = 0; k < S / 2; ++k) {
    const float keep = up ? a[k + S / 2] : a[k];
    const float send = up ? a[k] : a[k + S / 2];
    const float other = __shfl_xor_sync(0xffffffffu, send, 1 << bit);
    b[k] = MAX ? fmaxf(keep, other) : keep + other;
  }
}

// max or sum of each of the N columns over the warp's 32 rows (a
// reduce-scatter: 4 halving steps, then one exchange), written to dst[N]
template <int N, bool MAX>
__device__ __forceinline__ void colreduce(const float (&v)[N], int lane, float *dst) {
  float a1[N / 2], a2[N / 4], a3[N / 8], a4[N / 16];
  rs_half<N, MAX>(v, a1, lane, 4);
  rs_half<N / 2, MAX>(a1, a2, lane, 3);
  rs_half<N / 4, MAX>(a2, a3, lane, 2);
  rs_half<N / 8, MAX>(a3, a4, lane, 1);
#pragma unroll
  for (int k = 0; k < N / 16; ++k) {
    const float o = __shfl_xor_sync(0xffffffffu, a4[k], 1);
    a4[k] = MAX ? fmaxf(a4[k], o) : a4[k] + o;
  }
  if ((lane & 1) == 0) {
    const int base = ((lane >> 4) & 1) * (N / 2) + ((lane >> 3) & 1) * (N / 4) +
                     ((lane >> 2) & 1) * (N / 8) + ((lane >> 1) & 1) * (N / 16);
#pragma unroll
    for (int k = 0; k < N / 16; ++k) dst[base + k] = a4[k];
  }
}

// the same for any multiple of 8 columns: the reduce-scatter when the count
// is a multiple of 16, else a butterfly per column (lane 0 writes)
template <int N, bool MAX>
__device__ __forceinline__ void colreduce_any(const float (&v)[N], int lane, float *dst) {
  if constexpr (N % 16 == 0) {
    colreduce<N, MAX>(v, lane, dst);
  } else {
#pragma unroll
    for (int n = 0; n < N; ++n) {
      float x = v[n];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, o);
        x = MAX ? fmaxf(x, y) : x + y;
      }
      if (lane == 0) dst[n] = x;
    }
  }
}


// warps 8-11 (half 0) and 12-15 (half 1): token row t of each tile's S^T,
// columns (rows of the group) half * N/2 .. + N/2 - 1; per item an epilogue
// that writes O^T / l (thread t owns head-dim elements t and 128 + t of its
// rows)
template <int DT, int N>
__device__ void role_softmax(const AttnParams &p, uint8_t *smem, Ctl &c, uint32_t tmem,
                             int num_items, int warp, int lane, int half) {
  using Gm = Geo<DT, N>;
  constexpr float kRescale = 8.0f;
  // this warpgroup's columns (rows of the group): c0 .. c0 + NS - 1
  constexpr int NS = N / 2;
  const int c0 = half * NS;
  const uint32_t bar = half ? kBarSoftmax1 : kBarSoftmax;
  const int q4 = warp & 3, t = q4 * 32 + lane, jb = t >> 4;
  const uint32_t lb = tmem + ((uint32_t)(q4 * 32) << 16);
  const float qscale = p.scale_log2 * p.kv.kg;
  const float vg = p.kv.vg;
  // this thread's token column of P^T: chunk t / 64, 2-byte slot t % 8 of
  // 16-byte unit (t % 64) / 8, XORed with the row
  const uint32_t pcol = smem_u32(smem + Gm::OFF_P) + (t >> 6) * Gm::QCH + ((t & 7) << 1);
  const uint32_t s_m = smem_u32(c.m), s_lim = smem_u32(c.lim), s_inv = smem_u32(c.inv),
                 s_orow = smem_u32(c.orow);
  const int tu = (t & 63) >> 3;
  const int Hkv = p.kv.hkv;
  uint32_t g = 0, oi = 0;
  bool failed = false;
  for (int ii = blockIdx.x; ii < num_items && !failed; ii += gridDim.x) {
    const Item x = load_item(p, ii);
    const bool split = x.it.parts > 1;
    if (t < NS) {
      const int n = c0 + t;
      const bool live = n < x.R;
      const int qi = live ? (x.ro + n) / p.G : 0, gg = live ? (x.ro + n) % p.G : 0;
      c.lim[n] = live ? x.L - p.Q + 1 + qi : 0;
      c.orow[n] = split ? (x.it.slot * Hkv + x.kvh) * p.R + n
                        : (x.b * p.Q + qi) * p.Hq + x.kvh * p.G + gg;
      c.m[n] = kNegInf;
    }
    named_sync(bar, 128);
    // rows are written as fp32 (split-K partials or an fp32 output) or bf16
    const bool f32 = split || p.out_fp32;
    float *const of = split ? p.part_o : reinterpret_cast<float *>(p.out);
    __nv_bfloat16 *const ob = reinterpret_cast<__nv_bfloat16 *>(p.out);
    float *const lo = split ? p.part_lse : p.lse_out;
    const int R = x.R;
    // O^T columns (or zeros) of this group's rows for head-dim element d;
    // inv = 1 / l
    auto store_rows = [&](const float (&o)[NS], int d) {
#pragma unroll
      for (int n4 = 0; n4 < NS; n4 += 4) {
        const float4 iv = lds_f4(s_inv + 4 * (c0 + n4));
        const int4 rw = lds_s4(s_orow + 4 * (c0 + n4));
        const float ivs[4] = {iv.x, iv.y, iv.z, iv.w};
        const int rws[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (c0 + n4 + k < R) {
            const size_t off = (size_t)rws[k] * D + d;
            const float val = o[n4 + k] * ivs[k];
            if (f32) of[off] = val;
            else ob[off] = __float2bfloat16_rn(val);
          }
        }
      }
    };
    const bool empty = x.n_blk == 0;   // nothing to attend: zeros, lse -inf
    const int lim_min = x.L - p.Q + 1 + x.ro / p.G;   // the first live row's key limit
    float lp[NS];                                     // this row's share of each l
#pragma unroll
    for (int n = 0; n < NS; ++n) lp[n] = 0.f;
    for (int tile = 0; tile < x.ntiles; ++tile) {
      const int nb = min(kTileBlocks, x.n_blk - tile * kTileBlocks);
      const int tok0 = x.t_begin + tile * kTile, tok = tok0 + t;
      bool row_ok = jb < nb && tok < x.t_end;
      if (row_ok) {
        const int phys = x.trow[x.it.blk_begin + tile * kTileBlocks + jb];
        row_ok = phys >= 0 && phys < p.kv.num_blocks;
      }
      const bool causal = tok0 + kTile > lim_min;
      const int R = x.R;
      // log2-domain scores of one tile row (this thread's token), -inf where
      // masked; the causal limits are read only in the tiles that reach them
      auto scores = [&](float (&v)[NS]) {
#pragma unroll
        for (int n4 = 0; n4 < NS; n4 += 4) {
          int4 lm = make_int4(0x7fffffff, 0x7fffffff, 0x7fffffff, 0x7fffffff);
          if (causal) lm = lds_s4(s_lim + 4 * (c0 + n4));
          const int lv[4] = {lm.x, lm.y, lm.z, lm.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = n4 + k;
            const bool vis = row_ok && c0 + n < R && tok < lv[k];
            v[n] = vis ? v[n] * qscale : kNegInf;
          }
        }
      };
      const bool ok = wait_bar(&c.sfull[g & 1], (g >> 1) & 1, c, p.hdr) &&
                      wait_bar(&c.pdone[g & 1], ((g >> 1) & 1) ^ 1, c, p.hdr);
      tc_fence_after();
      const uint32_t sa = lb + kColS + (g & 1) * 64 + c0;
      const uint32_t pb = pcol + (g & 1) * Gm::PBUF;
      // Raw dot products in, probabilities out (written to P^T as f16) with
      // the running max m: p = 2^(s * scale - m), one FMA for the exponent;
      // `need` is set where a visible score passes m by the threshold.  The
      // exponent is capped so that a tile about to be redone stays finite.
      auto emit = [&](float (&v)[NS], bool &need) {
#pragma unroll
        for (int n4 = 0; n4 < NS; n4 += 4) {
          const float4 m4 = lds_f4(s_m + 4 * (c0 + n4));
          const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
          int4 lm = make_int4(0x7fffffff, 0x7fffffff, 0x7fffffff, 0x7fffffff);
          if (causal) lm = lds_s4(s_lim + 4 * (c0 + n4));
          const int lv[4] = {lm.x, lm.y, lm.z, lm.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = n4 + k, col = c0 + n;
            const bool vis = row_ok && col < R && tok < lv[k];
            const float d = fmaf(v[n], qscale, -mv[k]);
            need |= vis && d > kRescale;
            const float pr = vis ? ex2_approx(fminf(d, 64.f)) : 0.f;
            v[n] = pr;
            sts_u16(pb + col * 128 + ((tu ^ (col & 7)) << 4), __half_as_ushort(__float2half_rn(pr)));
          }
        }
      };
      // One pass with the current max; the first tile of an item (no max yet)
      // and the rare tile that raises a row's max by more than the threshold
      // are redone after the max update (a second pass of the same code).
      float v[NS];
      bool redo = tile == 0;
      bool stop = false;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (!redo || pass == 1) {   // probabilities with the current max
          tmem_ldn<NS>(sa, v);
          bool need = false;
          emit(v, need);
          if (pass == 1) break;
          redo = need;
        }
        if (!named_sync_or(bar, 128, redo || !ok)) break;
        if (named_sync_or(bar, 128, !ok)) {
          stop = true;
          break;
        }
        // new running max of every row: max over this tile's 128 rows
        tmem_ldn<NS>(sa, v);
        scores(v);
        colreduce_any<NS, true>(v, lane, c.red[q4] + c0);
        named_sync(bar, 128);
        if (t < NS) {
          const int n = c0 + t;
          const float mt = fmaxf(fmaxf(c.red[0][n], c.red[1][n]), fmaxf(c.red[2][n], c.red[3][n]));
          const float mo = c.m[n], mn = fmaxf(mo, mt);
          c.alpha[n] = mn == kNegInf ? 1.f : exp2f(mo - mn);
          c.mnew[n] = mn;
        }
        named_sync(bar, 128);
#pragma unroll
        for (int n = 0; n < NS; ++n) lp[n] *= c.alpha[c0 + n];
        if (tile > 0) {   // O^T holds this item's earlier tiles: rescale once PV(g-1) is done
          const bool ok2 = wait_bar(&c.pdone[(g - 1) & 1], ((g - 1) >> 1) & 1, c, p.hdr);
          if (named_sync_or(bar, 128, !ok2)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t oa = lb + kColO + c0;
#pragma unroll 1
          for (int hc = 0; hc < 2 * (NS / 8); ++hc) {   // (head-dim half, 8-column chunk)
            const int h = hc / (NS / 8), cb = hc % (NS / 8);
            float o[8];
            uint32_t w[8];
            tmem_ld8(oa + h * 64 + cb * 8, o);
#pragma unroll
            for (int k4 = 0; k4 < 8; k4 += 4) {
              const float4 a4 = lds_f4(smem_u32(c.alpha) + 4 * (c0 + cb * 8 + k4));
              w[k4] = __float_as_uint(o[k4] * a4.x);
              w[k4 + 1] = __float_as_uint(o[k4 + 1] * a4.y);
              w[k4 + 2] = __float_as_uint(o[k4 + 2] * a4.z);
              w[k4 + 3] = __float_as_uint(o[k4 + 3] * a4.w);
            }
            tmem_st8(oa + h * 64 + cb * 8, w);
          }
          tmem_st_wait();
        }
        if (t < NS) c.m[c0 + t] = c.mnew[c0 + t];
        named_sync(bar, 128);
        redo = true;
      }
      if (stop) {
        failed = true;
        break;
      }
#pragma unroll
      for (int n = 0; n < NS; ++n) lp[n] += v[n];   // this row's share of l
      tc_fence_before();
      mbar_arrive(&c.sfree[g & 1]);
      fence_async_smem();
      mbar_arrive(&c.pfull[g & 1]);
      ++g;
    }
    if (failed) break;
    // ---- epilogue: l of every row, then O^T / l (zeros for an empty item)
    colreduce_any<NS, false>(lp, lane, c.red[q4] + c0);
    const bool ok = empty || wait_bar(&c.odone, oi & 1, c, p.hdr);
    if (named_sync_or(bar, 128, !ok)) {
      failed = true;
      break;
    }
    if (t < NS) {
      const int n = c0 + t;
      const float l = (c.red[0][n] + c.red[1][n]) + (c.red[2][n] + c.red[3][n]);
      c.inv[n] = l > 0.f ? vg / l : 0.f;
      c.mnew[n] = l;
    }
    named_sync(bar, 128);
    tc_fence_after();
    const uint32_t oa = lb + kColO + c0;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float o[NS];
      if (!empty) {
        tmem_ldn<NS>(oa + h * 64, o);
      } else {
#pragma unroll
        for (int n = 0; n < NS; ++n) o[n] = 0.f;
      }
      store_rows(o, h * 128 + t);
    }
    if (t < NS && c0 + t < R && lo) {
      const int n = c0 + t;
      const float l = c.mnew[n];
      lo[c.orow[n]] = l > 0.f ? (c.m[n] + __log2f(l)) * 0.69314718055994531f : kNegInf;
    }
    if (!empty) {
      tc_fence_before();
      mbar_arrive(&c.ofree);
      ++oi;
    }
    named_sync(bar, 128);   // tables and sums read before the next item rewrites them
  }
}

template <int DT, int N>
__global__ void __launch_bounds__(kThreads, 1)
    verify_umma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  using Gm = Geo<DT, N>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ Ctl c;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  griddep_launch();   // the merge may start launching once every CTA has begun
  griddep_wait();     // the plan of this call is complete
  const int num_items = (int)p.hdr[HDR_NUM_ITEMS];
  if ((int)blockIdx.x >= num_items) return;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < Gm::NRK * kTileBlocks; ++s) {
      mbar_init(&c.rkfull[s], 1);
      mbar_init(&c.rkfree[s], kBlock);   // the block's 16 K rows
    }
#pragma unroll
    for (int s = 0; s < Gm::NRV * kTileBlocks; ++s) {
      mbar_init(&c.rvfull[s], 1);
      mbar_init(&c.rvfree[s], 2 * kBlock);   // the block's 16 V rows, two threads each
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mbar_init(&c.vfull[h], 128);   // every V thread
      mbar_init(&c.vfree[h], 1);     // the PV thread's commit
    }
    mbar_init(&c.ofree, 256);   // both softmax groups
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.sfull[i], 1);
      mbar_init(&c.sfree[i], 256);
      mbar_init(&c.pfull[i], 256);
      mbar_init(&c.pdone[i], 1);
      mbar_init(&c.kfull[i], 128);
      mbar_init(&c.kfree[i], 1);
    }
    mbar_init(&c.done, 2);   // one commit from each MMA-issuing thread
    mbar_init(&c.odone, 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem;

  const int wg = warp >> 2;   // warpgroup
  if (wg == 0) {
    setmaxnreg_to<kLaunchRegs, kRegCtl>();
    if (warp == 0 || warp == 3) {
      if (lane < kTileBlocks)
        role_producer<DT, N>(p, &tmK, &tmV, smem, c, num_items, lane, warp == 3 ? 1 : 0);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) role_qk<DT, N>(p, smem, c, tmem, num_items);
      __syncwarp();
    } else {
      if (lane == 0) role_pv<DT, N>(p, smem, c, tmem, num_items);
      __syncwarp();
    }
  } else if (wg == 1) {
    setmaxnreg_to<kLaunchRegs, kRegK>();
    role_kdeq<DT, N>(p, smem, c, tmem, num_items, warp, lane);
  } else if (wg == 2 || wg == 3) {
    setmaxnreg_to<kLaunchRegs, kRegSoftmax>();
    role_softmax<DT, N>(p, smem, c, tmem, num_items, warp, lane, wg - 2);
  } else {
    setmaxnreg_to<kLaunchRegs, kRegV>();
    role_vdeq<DT, N>(p, smem, c, num_items, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// grid: one persistent CTA per SM (never more than the planner's item bound)
template <int DT, int N>
cudaError_t launch_n(const AttnParams &p, int max_items, cudaStream_t s) {
  using Gm = Geo<DT, N>;
  auto kern = verify_umma_kernel<DT, N>;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)p.kv.num_blocks * p.kv.hkv * kBlock;
  if (!tc::make_row_map(&tk, p.kv.k, Gm::ROW, rows) || !tc::make_row_map(&tv, p.kv.v, Gm::ROW, rows))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
  if (e != cudaSuccess) return e;
  // the warpgroups' setmaxnreg steps start from kLaunchRegs: a build that
  // gave the kernel another count is refused, never launched
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidDeviceFunction;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = max(1, min(sms, max_items));
  return launch_pdl(kern, grid, kThreads, Gm::SMEM, s, p, tk, tv);
}

template <int DT>
cudaError_t launch_dtype(const AttnParams &p, int max_items, cudaStream_t s) {
  switch (p.R) {   // rows per group = the MMA's N
    case 16: return launch_n<DT, 16>(p, max_items, s);
    case 32: return launch_n<DT, 32>(p, max_items, s);
    case 48: return launch_n<DT, 48>(p, max_items, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace umma
}  // namespace pa
