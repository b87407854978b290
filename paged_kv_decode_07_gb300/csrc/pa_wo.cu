// pa_wo.cu -- the output projection after decode attention, in the same
// call: y[m, n] = sum_k o[m, k] * W[k, n], o the attention output of all
// query heads of a token flattened (k = head * D + d), W bf16 [Hq * D, N]
// ("vLLM Fork with focus on GB10 Homelabs", "Roadmap": fused attention +
// W_O GEMV, with a K-parallel split, CUTE_WO_SPLIT).
//
// At decode sizes (M = tokens <= a few dozen, K = Hq * D, N = hidden) the
// product streams W once: it is bound by HBM, not by arithmetic.  It runs on
// the tcgen05 tensor cores with the accumulators in tensor memory, in the
// transposed form y^T = W^T . o^T:
//   A = W^T [M = 128 hidden columns x K = 16] straight from the TMA boxes of
//       W (bf16, MN-major: W rows are k, contiguous in the hidden index);
//   B = o^T [K = 16 x N = 2 rows]: o is fp32 and enters as two bf16 terms,
//       hi = bf16(o) and lo = bf16(o - hi) (o - hi - lo is below 2^-16 |o|),
//       stacked as the N = 2 x rows columns of one K-major operand, so that one
//       MMA takes both terms; y = column r + column rows + r.
// W enters exactly.
//
// Grid: (N / 256 column tiles) x (k splits) x (64-row blocks of M), about
// one CTA per SM.  A CTA streams its W[k range, 256 columns] (four
// 64-column TMA boxes per 64-deep k chunk, 128-byte swizzle) and o[rows,
// k range] through a 4-stage mbarrier ring.  Warp 4 lane 0 issues the
// copies; warp 0 lane 0 issues, per chunk, 2 x 4 MMAs (two M = 128 tiles,
// four k16 steps) into two tensor-memory accumulators; warps 1-3 convert
// each o chunk into the bf16 hi / lo tiles (double-buffered) meanwhile;
// warps 0-3 read the accumulators at the end.  Copies and MMAs are issued
// by different threads because a chunk's six TMA instructions and its
// eight MMAs, issued by one thread, took about 1.7 K cycles per 40 KB
// chunk, which held the SM below a third of its share of DRAM bandwidth.
// Each o chunk is read once per 256 columns.
// Split partials go to the workspace and a second kernel adds them in fixed
// order (deterministic).  With programmatic dependent launch the W tiles of
// the first stages are requested before the attention's output is complete.
#include "pa_verify_umma.cuh"   // tcgen05 helpers (pa::umma)

namespace pa {
namespace {

constexpr int kWoThreads = 160;   // warp 0 MMAs, warps 1-3 conversion, warp 4 copies
constexpr int kWoConv = 96;       // converter threads (warps 1-3)
constexpr int kWoBoxN = 64;    // columns per TMA box of W (128 bytes of bf16)
constexpr int kWoBoxes = 4;    // boxes per chunk: 256 columns per CTA
constexpr int kWoN = kWoBoxes * kWoBoxN;
constexpr int kWoK = 64;       // k per chunk: four k16 steps
constexpr int kWoStages = 4;
constexpr int kWoRows = 64;    // rows of o per CTA at most (4 m16 tiles)
constexpr int kWoBoxBytes = kWoK * kWoBoxN * 2;      // 8 KB
constexpr int kWoWBytes = kWoBoxes * kWoBoxBytes;    // 32 KB
constexpr uint32_t kWoTmemCols = 256;   // two M = 128 tiles of up to N = 128 fp32 columns
// one 32-k fp32 box of o holds MT * 16 rows of 128 bytes
template <int MT>
struct WoGeo {
  static constexpr int ABox = MT * 16 * 128;
  static constexpr int Stage = kWoWBytes + 2 * ABox;   // multiple of 1024
  // the current chunk's o as bf16 hi and lo tiles [MT * 16 rows][64 k],
  // 128-byte rows with the 128-byte swizzle (conflict-free ldmatrix)
  static constexpr int XTile = MT * 16 * 128;
  // two X buffers (hi and lo tiles each), so that a chunk's conversion does
  // not wait for the previous chunk's MMAs
  static constexpr int Smem = kWoStages * Stage + 4 * XTile + 1024;
  static_assert(Stage % 1024 == 0, "swizzled boxes need 1024-byte alignment");
};

struct WoParams {
  const float *o;        // [M, K] fp32
  int M, K, N;
  int splits, chunks_per_split, ntiles;
  float *part;           // [splits, M, N] fp32 (splits > 1)
  void *y;               // [M, N]
  int y_fp32;
  uint32_t *hdr;
};

// (x0, x1) -> bf16x2 hi (x0 in the low half) and the bf16x2 of the remainders
__device__ __forceinline__ void split_bf16(float2 x, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x.x - hf.x, x.y - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// byte offset of fp32 (row, k) in a chunk's o tile: two boxes of 32 k
// (128-byte rows, 128-byte swizzle)
template <int MT>
__device__ __forceinline__ int a_off(int row, int k) {
  return (k >> 5) * WoGeo<MT>::ABox + row * 128 + (((((k & 31) * 4) >> 4) ^ (row & 7)) << 4) +
         ((k * 4) & 15);
}

// capped wait that also gives up once another thread of the CTA gave up
__device__ __forceinline__ bool wo_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
#pragma unroll 1
  for (uint32_t i = 0; i < kWaitCap; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

// Warp 4 lane 0 issues the copies, warp 0 lane 0 the MMAs; warps 1-3 turn
// each o chunk into the bf16 hi / lo tiles of the B operand.  Per chunk c
// (stage c % 4, X buffer c % 2):
//   full[st]  TMA -> converters (o box) and MMA thread (W boxes)
//   xfull[b]  converters -> MMA thread (96 arrivals)
//   xfree[b]  MMA commit -> converters (X b may be rewritten)
//   done[st]  MMA commit -> the copy thread's refill of stage st
// Warps 0-3 read the accumulators in the epilogue (warp w: lanes 32 w ..).
template <int MT>
__global__ void __launch_bounds__(kWoThreads, 1) wo_kernel(const WoParams p,
                                                           const __grid_constant__ CUtensorMap tmW,
                                                           const __grid_constant__ CUtensorMap tmA) {
  using namespace umma;
  using Gm = WoGeo<MT>;
  constexpr int kRows = MT * 16;       // rows of o per CTA
  constexpr int kN = 2 * kRows;        // MMA N: hi rows, then lo rows
  constexpr int kTiles = kWoN / 128;   // M = 128 column tiles of W per CTA
  constexpr int kConv = kWoConv;
  // instruction descriptor: D fp32, A and B bf16, A MN-major, B K-major
  constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                              ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static_assert(kN % 16 == 0 && kN <= 128, "MMA N (two tiles fit the tensor-memory columns)");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kWoStages], done[kWoStages], xfull[2], xfree[2], fin;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int *const abort = &s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockIdx.x % p.ntiles;
  const int s = (blockIdx.x / p.ntiles) % p.splits;
  const int mb = blockIdx.x / (p.ntiles * p.splits);
  const int n0 = nt * kWoN, m0 = mb * kWoRows;
  const int c0 = s * p.chunks_per_split;
  const int nch = max(0, min(p.chunks_per_split, p.K / kWoK - c0));
  // the column tiles of a split read the same o chunks: start each at a
  // different chunk so that they do not all hit the same L2 lines at once
  const int rot = nch > 0 ? (nt * 5) % nch : 0;

  const uint64_t pol = policy_evict_first();    // W: read once
  const uint64_t pol_o = policy_evict_last();   // o: read by every column tile
  auto chunk_k = [&](int c) { return (c0 + (c + rot) % nch) * kWoK; };
  auto issue = [&](int c, bool w_part, bool o_part) {   // the copy thread only
    uint8_t *st = smem + (c % kWoStages) * Gm::Stage;
    if (w_part) {
      mbar_arrive_expect_tx(&full[c % kWoStages], Gm::Stage);
#pragma unroll
      for (int w = 0; w < kWoBoxes; ++w)
        tc::tma_rows(st + w * kWoBoxBytes, &tmW, n0 + w * kWoBoxN, chunk_k(c),
                     &full[c % kWoStages], pol);
    }
    if (o_part) {   // o rows m0 .. m0 + 16 MT - 1, two 32-k boxes
      const int k = chunk_k(c);
      tc::tma_rows(st + kWoWBytes, &tmA, k, m0, &full[c % kWoStages], pol_o);
      tc::tma_rows(st + kWoWBytes + Gm::ABox, &tmA, k + 32, m0, &full[c % kWoStages], pol_o);
    }
  };
  const int pro = min(kWoStages, nch);
  if (tid == 128) {   // the copy thread: barriers, then the first W tiles at once
    for (int i = 0; i < kWoStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&done[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], kConv);
      mbar_init(&xfree[b], 1);
    }
    mbar_init(&fin, 1);
    fence_mbar_init();
    s_abort = 0;
    for (int c = 0; c < pro; ++c) issue(c, true, false);   // W does not depend on the attention
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, kWoTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  uint8_t *const xbase = smem + kWoStages * Gm::Stage;   // X[b]: hi rows then lo rows

  if (warp == 4) {
    if (lane == 0) {   // the copies (the first W tiles are in flight already)
      griddep_wait();   // o of this call is complete
      for (int c = 0; c < pro; ++c) issue(c, false, true);
      int issued = pro;
      // chunk c refills the stage of chunk c - 4 once its MMAs completed
      for (; issued < nch; ++issued) {
        const int pc = issued - kWoStages;
        if (!wo_wait(&done[pc % kWoStages], (pc / kWoStages) & 1, abort)) break;
        issue(issued, true, true);
      }
      // after a failure the copies still in flight (the last one of each
      // stage at most) land before the CTA exits
      if (*abort)
        for (int c = max(issued - kWoStages, 0); c < issued; ++c)
          (void)mbar_wait(&full[c % kWoStages], (c / kWoStages) & 1);
    }
    __syncwarp();
  } else if (warp == 0) {
    if (lane == 0) {   // the MMAs
      // descriptors are built once; an operand's start address (the low
      // field, address >> 4) moves by a constant per stage, tile and k step
      const uint64_t ad0 = sdesc(smem_u32(smem), kWoBoxBytes, 1024);
      const uint64_t bd0 = sdesc(smem_u32(xbase), 16, 1024);
      for (int c = 0; c < nch; ++c) {
        const int st = c % kWoStages;
        // both completion checks issued before either result is used
        const bool r1 = mbar_test(&full[st], (c / kWoStages) & 1);
        const bool r2 = mbar_test(&xfull[c & 1], (c >> 1) & 1);
        if (!(r1 || wo_wait(&full[st], (c / kWoStages) & 1, abort)) ||
            !(r2 || wo_wait(&xfull[c & 1], (c >> 1) & 1, abort)))
          break;
        tc_fence_after();
        const uint64_t wst = ad0 + (uint64_t)((st * Gm::Stage) >> 4);
        const uint64_t xb = bd0 + (uint64_t)(((c & 1) * 2 * Gm::XTile) >> 4);
#pragma unroll
        for (int mi = 0; mi < kTiles; ++mi)
#pragma unroll
          for (int ks = 0; ks < kWoK / 16; ++ks) {
            // A = W^T of columns 128 mi .. + 127 (two 64-column boxes LBO
            // apart, 8-row k groups 1024 bytes apart), chunk rows 16 ks .. + 15
            const uint64_t ad = wst + (uint64_t)((2 * mi * kWoBoxBytes + ks * 2048) >> 4);
            // B = [hi; lo] rows, k 16 ks .. + 15: 32 bytes into each 128-byte row
            const uint64_t bd = xb + (uint64_t)((ks * 32) >> 4);
            mma_ss(tmem + (uint32_t)(mi * kN), ad, bd, kIdesc, (c > 0 || ks > 0) ? 1u : 0u);
          }
        tc_commit(&done[st]);       // the stage may be refilled once these MMAs completed
        tc_commit(&xfree[c & 1]);   // and X[c % 2] rewritten
      }
      // every MMA complete before the accumulators are read (and released)
      tc_commit(&fin);
      (void)mbar_wait(&fin, 0);
      if (*abort) set_err(p.hdr, PA_ERRF_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
    // converters: o of chunk c -> bf16 hi and lo tiles, each element once per
    // CTA; thread i takes 8 consecutive k of one row (one 16-byte piece of each)
    const int ct = tid - 32;
    for (int c = 0; c < nch; ++c) {
      const int st = c % kWoStages;
      if (!wo_wait(&full[st], (c / kWoStages) & 1, abort)) break;
      if (c >= 2 && !wo_wait(&xfree[c & 1], ((c >> 1) - 1) & 1, abort)) break;
      const uint8_t *abase = smem + st * Gm::Stage + kWoWBytes;
      uint8_t *const xhi = xbase + (c & 1) * 2 * Gm::XTile, *const xlo = xhi + Gm::XTile;
      for (int i = ct; i < kRows * 8; i += kConv) {
        const int row = i >> 3, kc = i & 7;
        const float4 x0 = *reinterpret_cast<const float4 *>(abase + a_off<MT>(row, kc * 8));
        const float4 x1 = *reinterpret_cast<const float4 *>(abase + a_off<MT>(row, kc * 8 + 4));
        uint32_t hi[4], lo[4];
        split_bf16(make_float2(x0.x, x0.y), hi[0], lo[0]);
        split_bf16(make_float2(x0.z, x0.w), hi[1], lo[1]);
        split_bf16(make_float2(x1.x, x1.y), hi[2], lo[2]);
        split_bf16(make_float2(x1.z, x1.w), hi[3], lo[3]);
        const int off = row * 128 + ((kc ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(xhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(xlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_async_smem();   // generic-proxy writes of X -> visible to the tensor cores
      mbar_arrive(&xfull[c & 1]);
    }
  }
  __syncthreads();   // the MMA thread has seen `fin`
  tc_fence_after();
  if (!*abort && warp < 4) {
    // warp w reads tensor-memory lanes 32 w .. + 31: W columns n0 + 128 mi + 32 w + lane;
    // column r of the tile is token row r of hi, column kRows + r of lo
#pragma unroll 1
    for (int mi = 0; mi < kTiles; ++mi) {
      const int n = n0 + 128 * mi + 32 * warp + lane;
      const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(mi * kN);
      constexpr int kStep = kRows % 32 == 0 ? 32 : 16;   // rows per tensor-memory load
#pragma unroll 1
      for (int r0 = 0; r0 < kRows; r0 += kStep) {
        float h[kStep], l[kStep];
        if (nch > 0) {   // warp-uniform
          tmem_ldn<kStep>(ta + r0, h);
          tmem_ldn<kStep>(ta + kRows + r0, l);
        } else {
#pragma unroll
          for (int j = 0; j < kStep; ++j) h[j] = l[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < kStep; ++j) {
          const int m = m0 + r0 + j;
          if (m >= p.M || n >= p.N) continue;
          const float v = h[j] + l[j];
          if (p.splits > 1)
            p.part[((size_t)s * p.M + m) * p.N + n] = v;
          else if (p.y_fp32)
            static_cast<float *>(p.y)[(size_t)m * p.N + n] = v;
          else
            static_cast<__nv_bfloat16 *>(p.y)[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kWoTmemCols);
  }
}

// y = sum over splits of the partials, in split order; four consecutive
// elements per thread (all of a thread's loads in flight at once) where the
// buffers allow it, the rest one element per thread
__global__ void wo_reduce_kernel(const WoParams p) {
  griddep_wait();
  const size_t total = (size_t)p.M * p.N;
  // vector accesses only where every split's block and y are aligned for them
  const bool vec = total % 4 == 0 && reinterpret_cast<uintptr_t>(p.part) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(p.y) % (p.y_fp32 ? 16 : 8) == 0;
  const size_t n4 = vec ? total / 4 : 0;
  for (size_t i4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < n4;
       i4 += (size_t)gridDim.x * blockDim.x) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.splits; ++s) {
      const float4 x = reinterpret_cast<const float4 *>(p.part + (size_t)s * total)[i4];
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    if (p.y_fp32) {
      reinterpret_cast<float4 *>(p.y)[i4] = v;
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t *>(&lo);
      w.y = *reinterpret_cast<const uint32_t *>(&hi);
      reinterpret_cast<uint2 *>(p.y)[i4] = w;
    }
  }
  for (size_t i = 4 * n4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < p.splits; ++s) v += p.part[(size_t)s * total + i];
    if (p.y_fp32)
      static_cast<float *>(p.y)[i] = v;
    else
      static_cast<__nv_bfloat16 *>(p.y)[i] = __float2bfloat16_rn(v);
  }
}

bool make_map_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                 uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  tc::EncodeTiledFn fn = tc::encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT>
cudaError_t launch_mt(const WoParams &p, unsigned grid, const void *o, const CUtensorMap &tw,
                      cudaStream_t s) {
  CUtensorMap ta;
  std::memset(&ta, 0, sizeof ta);
  if (!make_map_2d(&ta, o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)p.K, (uint64_t)p.M, 32,
                   MT * 16))
    return cudaErrorInvalidValue;
  auto kern = wo_kernel<MT>;
  const int smem = WoGeo<MT>::Smem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, kWoThreads, smem, s, p, tw, ta);
}

}  // namespace

int wo_splits(int M, int K, int N, int requested) {
  const int chunks = K / kWoK;
  const int ntiles = (N + kWoN - 1) / kWoN;
  const int mblocks = (M + kWoRows - 1) / kWoRows;
  // about one CTA per SM (each holds a 4-stage ring of about 40-48 KB
  // stages, so one fits per SM); at least 4 chunks per split
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  int sp = requested > 0 ? requested : std::max(1, sms / (ntiles * mblocks));
  sp = std::max(1, std::min(sp, std::max(1, chunks / 4)));
  return std::min(sp, chunks);
}

cudaError_t launch_wo(const float *o, int M, int K, const void *w, int N, int splits, float *part,
                      void *y, int y_fp32, uint32_t *hdr, cudaStream_t s) {
  WoParams p;
  p.o = o;
  p.M = M;
  p.K = K;
  p.N = N;
  p.splits = splits;
  const int chunks = K / kWoK;
  p.chunks_per_split = (chunks + splits - 1) / splits;
  p.ntiles = (N + kWoN - 1) / kWoN;
  p.part = part;
  p.y = y;
  p.y_fp32 = y_fp32;
  p.hdr = hdr;
  CUtensorMap tw;
  std::memset(&tw, 0, sizeof tw);
  if (!make_map_2d(&tw, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)N, (uint64_t)K, kWoBoxN,
                   kWoK))
    return cudaErrorInvalidValue;
  const int mblocks = (M + kWoRows - 1) / kWoRows;
  const unsigned grid = (unsigned)(p.ntiles * splits * mblocks);
  const int rows = std::min(M, kWoRows);
  cudaError_t e = rows > 32 ? launch_mt<4>(p, grid, o, tw, s)
                  : rows > 16 ? launch_mt<2>(p, grid, o, tw, s)
                              : launch_mt<1>(p, grid, o, tw, s);
  if (e != cudaSuccess || splits == 1) return e;
  const size_t total = (size_t)M * N;
  const unsigned rgrid = (unsigned)std::min<size_t>((total / 4 + 255) / 256 + 1, 2048);
  return launch_pdl(wo_reduce_kernel, rgrid, 256, 0, s, p);
}

}  // namespace pa
