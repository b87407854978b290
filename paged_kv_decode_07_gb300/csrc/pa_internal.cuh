// pa_internal.cuh -- shared device-side definitions of the paged-KV decode
// library (sm_103a).  Not part of the public ABI (include/pa.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pa.h"

namespace pa {

constexpr int kBlock = 16;            // tokens per KV block
constexpr int kMaxG = 8;              // query heads per kv head handled in one item
constexpr int kMaxQLen = 16;
constexpr int kHdrWords = 64;         // 256-byte workspace header
constexpr int kMaxTargetItems = 4096;
// work items the planner aims at when the caller names no target: about 8
// per SM for the one-CTA-per-item decode kernels
constexpr int kDefaultTargetItems = 1184;
constexpr uint32_t kWaitCap = 1u << 22;   // iteration cap of every in-kernel wait
constexpr uint32_t kTestWaitCap = 1u << 10;   // cap of the waits a PA_TEST_EXPIRE_WAIT call expires
constexpr float kNegInf = -__builtin_huge_valf();

// workspace header words
enum : int {
  HDR_ERR = 0,         // PA_ERRF_* bits of the current call
  HDR_NUM_ITEMS = 1,   // work items planned
  HDR_SPLIT = 2,       // blocks per partition chosen by the planner
  HDR_NUM_SLOTS = 3,   // partial slots used
  HDR_ROUND = 4,       // resident CTAs the item count was rounded to (0: not rounded)
};

// KV pool as the kernels see it
struct KvView {
  int dtype, num_blocks, hkv, D;
  const void *k, *v, *ks, *vs;
  float kg, vg;
};

// A plan "unit" is a (sequence, query-row group).  Mode 1 (virtual): one
// unit per (b, i) query token with its own key limit; mode 0 (dense): one
// unit per sequence holding all q_len * G rows; mode 2 (row groups): one
// unit per (b, group of R consecutive rows of the q_len * G), R a multiple
// of 16 up to kMaxRowGroup.
constexpr int kMaxRowGroup = 48;
struct UnitInfo {      // int4 in the workspace
  int parts;           // partitions (0 = nothing to attend)
  int slot_base;       // first partial slot (parts > 1), else -1
  int nblk;            // key blocks covered
  int len;             // key limit of the unit (max over its rows)
};

struct WorkItem {      // two int4 in the workspace
  int unit, kvh, blk_begin, blk_end;
  int part, parts, slot, pad;
};

// Everything an attention kernel needs; passed by value.
struct AttnParams {
  KvView kv;
  const __nv_bfloat16 *q;   // [B, Q, Hq, D]
  int B, Q, Hq, G;
  const int *tables;
  int stride;
  const int *seq_lens;
  float scale_log2;         // softmax_scale * log2(e)
  void *out;
  int out_fp32;
  float *lse_out;
  // plan
  uint32_t *hdr;
  const WorkItem *items;
  const UnitInfo *units;
  float *part_o;            // [slot][Hkv][R][D]
  float *part_lse;          // [slot][Hkv][R]
  int max_items;
  int max_slots;
  int virt;                 // plan mode: 1 virtual, 0 dense, 2 row groups
  int R;                    // rows per item: G (virtual), Q*G (dense), rows per group (mode 2)
  int RG;                   // row groups per sequence (mode 2), else 1
  int test_expire;          // PA_TEST_EXPIRE_WAIT: first copies withheld, short wait cap
};

struct PlanParams {
  const int *seq_lens;
  int B, Q, virt, hkv;
  int RG;                   // row groups per sequence (mode 2), else 1
  int capacity;             // 16 * stride
  int target_items, split_blocks, min_split_blocks;
  int max_items, max_slots;
  // CTAs of the attention kernel resident at once on the whole GPU (SMs x
  // CTAs per SM), or 0: with equal-length sequences the planner then makes
  // the item count a whole number of such rounds; item_cost is the fixed
  // cost of one item in key blocks streamed, which sets how many rounds
  int resident, item_cost;
  uint32_t *hdr;
  WorkItem *items;
  UnitInfo *units;
  int *prefix_a, *prefix_b; // [units] scratch
  const uint32_t *extra_err; // flags of an earlier kernel of the same call, or null
};

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// true when the phase with the given parity has completed
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait; false if the cap was hit
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint32_t cap = kWaitCap) {
  for (uint32_t i = 0; i < cap; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared (TMA engine), completion on an mbarrier.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch: a kernel launched with the
// programmatic-serialization attribute may start before its predecessor in
// the stream finishes; griddep_wait() blocks until the predecessor has
// completed and its memory is visible (a no-op without the attribute).
// griddep_launch() lets the next kernel in the stream start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kern` so that it may overlap the tail of the previous kernel in
// the stream (it must call griddep_wait() before touching that kernel's
// results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void set_err(uint32_t *hdr, uint32_t bits) {
  if (hdr) atomicOr(hdr + HDR_ERR, bits);
}

// -------------------------------------------------------- format decoding

// two bf16 packed in a u32 -> (lo, hi) fp32, exact
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// four int8 codes in a u32 -> fp32 values, exact: place (code ^ 0x80) in the
// low byte of 2^23 and subtract 2^23 + 128.
__device__ __forceinline__ void s8x4_to_f4(uint32_t u, float *o) {
  uint32_t x = u ^ 0x80808080u;
  const float bias = 8388736.0f;   // 2^23 + 128
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t bits = __byte_perm(x, 0x4B000000u, 0x7640 | j);
    o[j] = __uint_as_float(bits) - bias;
  }
}

// one byte of two E2M1 codes -> f16x2 (low nibble in .x), exact
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// E4M3 byte -> f16x2 with the value in both halves, exact
__device__ __forceinline__ uint32_t e4m3_to_h2_dup(uint32_t byte) {
  uint32_t r;
  uint16_t pair = (uint16_t)(byte | (byte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}

// two E4M3 codes (low 16 bits, element 0 in the low byte) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_u16_to_h2(uint32_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v));
  return r;
}

__device__ __forceinline__ constexpr bool has_scale_tensors(int dt) {
  return dt == PA_KV_INT8 || dt == PA_KV_NVFP4;
}
__device__ __forceinline__ constexpr bool has_global_scale(int dt) {
  return dt == PA_KV_NVFP4 || dt == PA_KV_FP8;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ float2 h2u_to_f2(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2 *>(&u));
}

__device__ __forceinline__ float fp16_bits_to_f(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// --------------------------------------------------------- f32x2 arithmetic

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(*reinterpret_cast<unsigned long long *>(&d))
      : "l"(*reinterpret_cast<unsigned long long *>(&a)),
        "l"(*reinterpret_cast<unsigned long long *>(&b)),
        "l"(*reinterpret_cast<unsigned long long *>(&c)));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long *>(&d))
      : "l"(*reinterpret_cast<unsigned long long *>(&a)),
        "l"(*reinterpret_cast<unsigned long long *>(&b)));
  return d;
}

}  // namespace pa
