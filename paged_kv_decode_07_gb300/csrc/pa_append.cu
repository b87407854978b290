// pa_append.cu -- quantise-on-write of new tokens' K and V into the paged
// pool: the write side of PagedAttention (Kwon et al., cited on "vLLM Fork
// with focus on GB10 Homelabs", "About"): token t's rows go to the slot
// slot_mapping[t] = physical block * 16 + offset, and a padded row carries
// slot -1 and writes nothing ("vLLM-SM70", "Known limitations": padded
// drafter rows once wrote K/V into other requests' slots).
//
// Each warp takes four consecutive (token, kv head) rows; their K and V
// (D bf16 each, 16 or 8 bytes per lane, coalesced) are loaded together,
// encoded in registers and written as one contiguous code run per row.
// NVFP4 gives each lane one 16-element scale block instead (two or four
// rows per warp step).  Every rounding decision is
// that of the IEEE fp32 quotient (formed without a division per element,
// see the bracket below), so the codes are the format definitions' own:
//   int8  : s = fp16_RN(amax / 127), code = clamp(RN_even(x / s), +-127)
//   FP8   : code = E4M3_RN_satfinite(|x / g|) with the sign of x / g unless
//           the magnitude code is 0
//   NVFP4 : per 16 elements, scale = E4M3_RN_satfinite(amax16 / (g * 6)),
//           code = E2M1_RN_satfinite(|x / (e4m3(scale) * g)|) | sign << 3,
//           element 2i in the low nibble
//   bf16  : copied
// The conversions to fp16 / E4M3 / E2M1 are the hardware's round-to-nearest
// (satfinite) cvt instructions on signed values; the FP8 rule for zero is
// applied to the packed codes afterwards.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kAppendWarps = 8;

struct AppendParams {
  KvView kv;
  const __nv_bfloat16 *k_new, *v_new;   // [T, Hkv, D]
  const int64_t *slots;                 // [T]
  int T;
  uint32_t *hdr;                        // may be null
};

// (lo, hi) -> two E4M3 codes, lo in the low byte; round to nearest even,
// saturating at 448
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// eight magnitudes -> eight E2M1 codes, element 2i in the low nibble of byte i
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(const float (&a)[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(r)
      : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
  return r;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  return __half2float(__ushort_as_half((uint16_t)(e4m3x2_u16_to_h2(code) & 0xFFFFu)));
}

template <int EPL>
struct Chunk {   // EPL bf16 of one lane
  uint32_t w[EPL / 2];
};

template <int EPL>
__device__ __forceinline__ Chunk<EPL> load_chunk(const __nv_bfloat16 *p) {
  Chunk<EPL> c;
  if constexpr (EPL == 8) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
    c.w[0] = u.x; c.w[1] = u.y; c.w[2] = u.z; c.w[3] = u.w;
  } else {
    const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p));
    c.w[0] = u.x; c.w[1] = u.y;
  }
  return c;
}

template <int EPL>
__device__ __forceinline__ void to_float(const Chunk<EPL> &c, float (&x)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL / 2; ++i) {
    const float2 f = bf16x2_to_f2(c.w[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// ---- quotients without a division per element.  With r an approximate
// reciprocal of the divisor d (rcp.approx, at most 1 ulp off, i.e. a
// relative error below 2^-23), RN(x * r) lies within 2^-22 of the IEEE
// quotient RN(x / d), relatively.  Rounding onto a grid (integers, fp16,
// E4M3, E2M1) is monotone, so the decision is taken at both ends of a
// bracket that must hold the exact quotient -- x * RN(r * (1 -+ 2^-20)) --
// and when the two ends agree that is the decision of RN(x / d) itself.
// Otherwise (a few in 10^5 elements) the quotient is formed exactly.  For
// int8 the bracket is the distance to the nearest half integer instead:
// |x / d| < 2^8 there, so RN(x * r) is within 2^-14 of RN(x / d) and a
// margin of 2^-13 decides.
constexpr float kBracketLo = 1.0f - 0x1p-20f;
constexpr float kBracketHi = 1.0f + 0x1p-20f;
constexpr float kInf = __builtin_huge_valf();

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long *>(&d))
      : "l"(*reinterpret_cast<unsigned long long *>(&a)),
        "l"(*reinterpret_cast<unsigned long long *>(&b)));
  return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long *>(&d))
      : "l"(*reinterpret_cast<unsigned long long *>(&a)),
        "l"(*reinterpret_cast<unsigned long long *>(&b)));
  return d;
}

// low bytes of four words -> one word
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// E4M3 codes of RN(x / d) for EPL values, 4 per word; `ok` = false when the
// bracket could not decide (the caller then forms exact quotients)
template <int EPL>
__device__ __forceinline__ void e4m3_codes(const float (&x)[EPL], float rlo, float rhi,
                                           uint32_t (&w)[EPL / 4], bool &ok) {
#pragma unroll
  for (int k = 0; k < EPL / 4; ++k) {
    const float2 a = fmul2(make_float2(x[4 * k], x[4 * k + 1]), make_float2(rlo, rlo));
    const float2 b = fmul2(make_float2(x[4 * k + 2], x[4 * k + 3]), make_float2(rlo, rlo));
    const float2 c = fmul2(make_float2(x[4 * k], x[4 * k + 1]), make_float2(rhi, rhi));
    const float2 e = fmul2(make_float2(x[4 * k + 2], x[4 * k + 3]), make_float2(rhi, rhi));
    const uint32_t lo = __byte_perm(e4m3x2_rn_sat(a.x, a.y), e4m3x2_rn_sat(b.x, b.y), 0x5410u);
    const uint32_t hi = __byte_perm(e4m3x2_rn_sat(c.x, c.y), e4m3x2_rn_sat(e.x, e.y), 0x5410u);
    ok = ok && lo == hi;
    w[k] = lo;
  }
}

// a byte whose magnitude bits are 0 is written +0
__device__ __forceinline__ uint32_t plus_zero(uint32_t w) {
  const uint32_t nz = (w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;   // bit 7 set iff magnitude != 0
  return w & (nz | 0x7F7F7F7Fu);
}

template <int DT, int D>
__device__ __forceinline__ void encode_store(const AppendParams &p, int which, size_t row,
                                             const Chunk<D / 32> &c, int lane) {
  constexpr int EPL = D / 32;
  void *data = const_cast<void *>(which ? p.kv.v : p.kv.k);
  void *scale = const_cast<void *>(which ? p.kv.vs : p.kv.ks);
  if constexpr (DT == PA_KV_BF16) {
    uint8_t *dst = static_cast<uint8_t *>(data) + (row * D + lane * EPL) * 2;
    if constexpr (EPL == 8)
      *reinterpret_cast<uint4 *>(dst) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
    else
      *reinterpret_cast<uint2 *>(dst) = make_uint2(c.w[0], c.w[1]);
    return;
  } else {
    float x[EPL];
    to_float<EPL>(c, x);
    uint32_t w[EPL / 4];   // EPL one-byte codes (int8, FP8) or EPL nibbles (NVFP4)
    if constexpr (DT == PA_KV_INT8) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // s = fp16_RN(RN(amax / 127)), amax the same in every lane
      constexpr float r127 = 1.0f / 127.0f;
      __half s16 = __float2half_rn(__fmul_rn(amax, r127 * kBracketLo));
      if (__half_as_ushort(s16) != __half_as_ushort(__float2half_rn(__fmul_rn(amax, r127 * kBracketHi))))
        s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
      const float s = __half2float(s16);
      const float rs = rcp_approx(s);
      constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: adding it rounds to an integer (RNE)
      const bool clamp = s < 0x1p-14f;        // fp16-subnormal scale: |x / s| may pass 127.5
      bool near = false;
      float t[EPL];
#pragma unroll
      for (int i = 0; i < EPL; i += 2) {
        float2 q = fmul2(make_float2(x[i], x[i + 1]), make_float2(rs, rs));
        if (clamp) {
          q.x = fminf(fmaxf(q.x, -127.f), 127.f);
          q.y = fminf(fmaxf(q.y, -127.f), 127.f);
        }
        const float2 tt = fadd2(q, make_float2(kMagic, kMagic));              // rint(q) + M
        const float2 f = fsub2(q, fsub2(tt, make_float2(kMagic, kMagic)));   // q - rint(q), exact
        near = near || fabsf(f.x) > 0.5f - 0x1p-13f || fabsf(f.y) > 0.5f - 0x1p-13f;
        t[i] = tt.x;
        t[i + 1] = tt.y;
      }
#pragma unroll
      for (int k = 0; k < EPL / 4; ++k)   // rint(q) mod 256 is the low byte of rint(q) + M
        w[k] = low_bytes(__float_as_uint(t[4 * k]), __float_as_uint(t[4 * k + 1]),
                         __float_as_uint(t[4 * k + 2]), __float_as_uint(t[4 * k + 3]));
      if (__any_sync(0xffffffffu, near) && near) {   // next to a half integer: exact quotients
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) {
          uint32_t b[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            b[j] = (uint32_t)max(-127, min(127, __float2int_rn(__fdiv_rn(x[4 * k + j], s))));
          w[k] = low_bytes(b[0], b[1], b[2], b[3]);
        }
      }
      if (!(s > 0.f)) {
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) w[k] = 0;
      }
      if (lane == 0) static_cast<__half *>(scale)[row] = s16;
    } else if constexpr (DT == PA_KV_FP8) {
      const float g = which ? p.kv.vg : p.kv.kg;
      const float rg = rcp_approx(g);
      bool ok = g > 0.f && rg < kInf;
      e4m3_codes<EPL>(x, __fmul_rn(rg, kBracketLo), __fmul_rn(rg, kBracketHi), w, ok);
      if (__any_sync(0xffffffffu, !ok) && !ok) {
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) {
          float y[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) y[j] = g > 0.f ? __fdiv_rn(x[4 * k + j], g) : 0.f;
          w[k] = __byte_perm(e4m3x2_rn_sat(y[0], y[1]), e4m3x2_rn_sat(y[2], y[3]), 0x5410u);
        }
      }
#pragma unroll
      for (int k = 0; k < EPL / 4; ++k) w[k] = plus_zero(w[k]);
    } else {   // NVFP4: a 16-element scale block spans 16 / EPL lanes
      const float g = which ? p.kv.vg : p.kv.kg;
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int o = 1; o < 16 / EPL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // block scale = E4M3(RN(amax / RN(g * 6)))
      const float den = __fmul_rn(g, 6.0f);
      const float rden = rcp_approx(den);
      uint32_t sc = e4m3x2_rn_sat(__fmul_rn(amax, __fmul_rn(rden, kBracketLo)), 0.f) & 0xFFu;
      const uint32_t sc_hi = e4m3x2_rn_sat(__fmul_rn(amax, __fmul_rn(rden, kBracketHi)), 0.f) & 0xFFu;
      if (!(g > 0.f && rden < kInf) || sc != sc_hi)
        sc = g > 0.f ? (e4m3x2_rn_sat(__fdiv_rn(amax, den), 0.f) & 0xFFu) : 0u;
      const float sg = __fmul_rn(e4m3_to_float(sc), g);
      const float rsg = rcp_approx(sg);
      const float rlo = __fmul_rn(rsg, kBracketLo), rhi = __fmul_rn(rsg, kBracketHi);
      float lo[8], hi[8];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float2 xx = i < EPL ? make_float2(x[i], x[i + 1]) : make_float2(0.f, 0.f);
        const float2 a = fmul2(xx, make_float2(rlo, rlo)), b = fmul2(xx, make_float2(rhi, rhi));
        lo[i] = a.x; lo[i + 1] = a.y;
        hi[i] = b.x; hi[i + 1] = b.y;
      }
      // signed inputs: the code's sign bit is that of x / sg, -0 included
      uint32_t codes = e2m1x8_rn_sat(lo);
      const bool ok = sg > 0.f && rsg < kInf && codes == e2m1x8_rn_sat(hi);
      if (__any_sync(0xffffffffu, !ok) && !ok) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = (i < EPL && sg > 0.f) ? __fdiv_rn(x[i], sg) : 0.f;
        codes = e2m1x8_rn_sat(y);
      }
      if (!(sg > 0.f)) codes = 0;   // the quotient is taken as +0
      w[0] = codes;
      if ((lane & (16 / EPL - 1)) == 0)
        static_cast<uint8_t *>(scale)[row * (D / 16) + lane * EPL / 16] = (uint8_t)sc;
    }
    // ---- store the codes
    if constexpr (DT == PA_KV_NVFP4) {
      uint8_t *dst = static_cast<uint8_t *>(data) + row * (D / 2) + lane * (EPL / 2);
      if constexpr (EPL == 8)
        *reinterpret_cast<uint32_t *>(dst) = w[0];
      else
        *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w[0];
    } else {
      uint8_t *dst = static_cast<uint8_t *>(data) + row * D + lane * EPL;
      if constexpr (EPL == 8)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    }
  }
}

// kRows consecutive (token, kv head) rows per warp: their slots and K / V
// chunks are all loaded before the first is encoded, so that a warp keeps
// kRows * 2 * D * 2 bytes in flight (padded rows are read and dropped).
constexpr int kRows = 4;

template <int DT, int D>
__global__ void __launch_bounds__(kAppendWarps * 32, 4) append_kernel(const AppendParams p) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  // rows < 2^30 (checked on the host): 32-bit indices, one division per warp
  const int r0 = (blockIdx.x * kAppendWarps + (threadIdx.x >> 5)) * kRows;
  const int Hkv = p.kv.hkv;
  const int nrows = p.T * Hkv;
  if (r0 >= nrows) return;
  int64_t slot[kRows];
  int head[kRows];
  Chunk<EPL> ck[kRows], cv[kRows];
  int t = r0 / Hkv, h = r0 - t * Hkv;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const int r = r0 + j;
    head[j] = h;
    if (r < nrows) {
      slot[j] = __ldg(p.slots + t);
      const size_t src = (size_t)r * D + lane * EPL;
      ck[j] = load_chunk<EPL>(p.k_new + src);
      cv[j] = load_chunk<EPL>(p.v_new + src);
    } else {
      slot[j] = -1;
    }
    if (++h == Hkv) {
      h = 0;
      ++t;
    }
  }
  const int64_t nslots = (int64_t)p.kv.num_blocks * kBlock;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    if (slot[j] == -1) continue;   // padded row (or past the end)
    if (slot[j] < -1 || slot[j] >= nslots) {
      if (lane == 0) set_err(p.hdr, PA_ERRF_BAD_SLOT);
      continue;
    }
    const int blk = (int)(slot[j] >> 4), off = (int)slot[j] & (kBlock - 1);
    const size_t row = ((size_t)blk * Hkv + head[j]) * kBlock + off;
    encode_store<DT, D>(p, 0, row, ck[j], lane);
    encode_store<DT, D>(p, 1, row, cv[j], lane);
  }
}

// ---- NVFP4 with one 16-element scale block per lane: D / 16 lanes per row
// and 512 / D rows per warp step, so the block max needs no shuffle and the
// scale work (bracketed E4M3 scale, reciprocal) is shared by 16 elements.
// The decisions are those of encode_store<PA_KV_NVFP4> above.
__device__ __forceinline__ void nvfp4_encode16(const uint4 (&u)[2], float g, bool store,
                                               uint8_t *cdst, uint8_t *sdst) {
  const uint32_t wv[8] = {u[0].x, u[0].y, u[0].z, u[0].w, u[1].x, u[1].y, u[1].z, u[1].w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = bf16x2_to_f2(wv[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  // block scale = E4M3(RN(amax / RN(g * 6)))
  const float den = __fmul_rn(g, 6.0f);
  const float rden = rcp_approx(den);
  uint32_t sc = e4m3x2_rn_sat(__fmul_rn(amax, __fmul_rn(rden, kBracketLo)), 0.f) & 0xFFu;
  const uint32_t sc_hi = e4m3x2_rn_sat(__fmul_rn(amax, __fmul_rn(rden, kBracketHi)), 0.f) & 0xFFu;
  if (!(g > 0.f && rden < kInf) || sc != sc_hi)
    sc = g > 0.f ? (e4m3x2_rn_sat(__fdiv_rn(amax, den), 0.f) & 0xFFu) : 0u;
  const float sg = __fmul_rn(e4m3_to_float(sc), g);
  const float rsg = rcp_approx(sg);
  const float rlo = __fmul_rn(rsg, kBracketLo), rhi = __fmul_rn(rsg, kBracketHi);
  float lo0[8], lo1[8], hi0[8], hi1[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 a = fmul2(make_float2(x[i], x[i + 1]), make_float2(rlo, rlo));
    const float2 b = fmul2(make_float2(x[i], x[i + 1]), make_float2(rhi, rhi));
    const float2 c = fmul2(make_float2(x[8 + i], x[9 + i]), make_float2(rlo, rlo));
    const float2 d = fmul2(make_float2(x[8 + i], x[9 + i]), make_float2(rhi, rhi));
    lo0[i] = a.x; lo0[i + 1] = a.y;
    hi0[i] = b.x; hi0[i + 1] = b.y;
    lo1[i] = c.x; lo1[i + 1] = c.y;
    hi1[i] = d.x; hi1[i + 1] = d.y;
  }
  // signed inputs: the code's sign bit is that of x / sg, -0 included
  uint32_t c0 = e2m1x8_rn_sat(lo0), c1 = e2m1x8_rn_sat(lo1);
  const bool ok = sg > 0.f && rsg < kInf && c0 == e2m1x8_rn_sat(hi0) && c1 == e2m1x8_rn_sat(hi1);
  if (__any_sync(0xffffffffu, !ok) && !ok) {
    float y0[8], y1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y0[i] = sg > 0.f ? __fdiv_rn(x[i], sg) : 0.f;
      y1[i] = sg > 0.f ? __fdiv_rn(x[8 + i], sg) : 0.f;
    }
    c0 = e2m1x8_rn_sat(y0);
    c1 = e2m1x8_rn_sat(y1);
  }
  if (!(sg > 0.f)) c0 = c1 = 0;   // the quotient is taken as +0
  if (store) {
    *reinterpret_cast<uint2 *>(cdst) = make_uint2(c0, c1);
    *sdst = (uint8_t)sc;
  }
}

// 3 CTAs per SM: the 8 K / V chunks a lane keeps in flight need more than 64 registers
template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32, 3) append_nvfp4_kernel(const AppendParams p) {
  constexpr int LPR = D / 16, RPS = 32 / LPR, STEPS = kRows / RPS;
  static_assert(STEPS >= 1 && kRows % RPS == 0, "rows per warp");
  const int lane = threadIdx.x & 31, sub = lane / LPR, ll = lane % LPR;
  // rows < 2^30 (checked on the host): 32-bit indices
  const int r0 = (blockIdx.x * kAppendWarps + (threadIdx.x >> 5)) * kRows;
  const int Hkv = p.kv.hkv;
  const int nrows = p.T * Hkv;
  if (r0 >= nrows) return;   // the whole warp: every lane below runs the same steps
  int64_t slot[STEPS];
  int head[STEPS];
  uint4 kx[STEPS][2], vx[STEPS][2];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int r = r0 + s * RPS + sub;
    const int t = r / Hkv;
    head[s] = r - t * Hkv;
    if (r < nrows) {
      slot[s] = __ldg(p.slots + t);
      const size_t src = (size_t)r * D + ll * 16;
      kx[s][0] = __ldcs(reinterpret_cast<const uint4 *>(p.k_new + src));
      kx[s][1] = __ldcs(reinterpret_cast<const uint4 *>(p.k_new + src + 8));
      vx[s][0] = __ldcs(reinterpret_cast<const uint4 *>(p.v_new + src));
      vx[s][1] = __ldcs(reinterpret_cast<const uint4 *>(p.v_new + src + 8));
    } else {
      slot[s] = -1;
      kx[s][0] = kx[s][1] = vx[s][0] = vx[s][1] = make_uint4(0, 0, 0, 0);
    }
  }
  const int64_t nslots = (int64_t)p.kv.num_blocks * kBlock;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const bool bad = slot[s] < -1 || slot[s] >= nslots;
    if (bad && ll == 0) set_err(p.hdr, PA_ERRF_BAD_SLOT);
    const bool st = slot[s] >= 0 && !bad;   // -1: padded row (or past the end)
    size_t row = 0;
    if (st) {
      const int blk = (int)(slot[s] >> 4), off = (int)slot[s] & (kBlock - 1);
      row = ((size_t)blk * Hkv + head[s]) * kBlock + off;
    }
    nvfp4_encode16(kx[s], p.kv.kg, st, static_cast<uint8_t *>(const_cast<void *>(p.kv.k)) + row * (D / 2) + ll * 8,
                   static_cast<uint8_t *>(const_cast<void *>(p.kv.ks)) + row * (D / 16) + ll);
    nvfp4_encode16(vx[s], p.kv.vg, st, static_cast<uint8_t *>(const_cast<void *>(p.kv.v)) + row * (D / 2) + ll * 8,
                   static_cast<uint8_t *>(const_cast<void *>(p.kv.vs)) + row * (D / 16) + ll);
  }
}

template <int DT>
cudaError_t launch_dt(const AppendParams &p, cudaStream_t s) {
  const int rows = p.T * p.kv.hkv;
  const int per_cta = kAppendWarps * kRows;
  const unsigned grid = (unsigned)((rows + per_cta - 1) / per_cta);
  if constexpr (DT == PA_KV_NVFP4) {
    if (p.kv.D == 128)
      append_nvfp4_kernel<128><<<grid, kAppendWarps * 32, 0, s>>>(p);
    else
      append_nvfp4_kernel<256><<<grid, kAppendWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
  }
  if (p.kv.D == 128)
    append_kernel<DT, 128><<<grid, kAppendWarps * 32, 0, s>>>(p);
  else
    append_kernel<DT, 256><<<grid, kAppendWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const KvView &kv, const void *k_new, const void *v_new, int T,
                          const int64_t *slots, uint32_t *hdr, cudaStream_t s) {
  AppendParams p;
  p.kv = kv;
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.slots = slots;
  p.T = T;
  p.hdr = hdr;
  switch (kv.dtype) {
    case PA_KV_BF16: return launch_dt<PA_KV_BF16>(p, s);
    case PA_KV_INT8: return launch_dt<PA_KV_INT8>(p, s);
    case PA_KV_NVFP4: return launch_dt<PA_KV_NVFP4>(p, s);
    case PA_KV_FP8: return launch_dt<PA_KV_FP8>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
