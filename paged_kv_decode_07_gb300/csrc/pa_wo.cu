// pa_wo.cu -- the output projection after decode attention, in the same
// call: y[m, n] = sum_k o[m, k] * W[k, n], o the attention output of all
// query heads of a token flattened (k = head * D + d), W bf16 [Hq * D, N]
// ("vLLM Fork with focus on GB10 Homelabs", "Roadmap": fused attention +
// W_O GEMV, with a K-parallel split, CUTE_WO_SPLIT).
//
// At decode sizes (M = tokens <= a few dozen, K = Hq * D, N = hidden) the
// product streams W once: it is bound by HBM, not by arithmetic, and runs
// on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32
// accumulation) so that the issue slots stay free for the copies.  o is
// fp32; it enters the MMA as two bf16 terms hi = bf16(o), lo = bf16(o - hi)
// (o - hi - lo is below 2^-16 |o|), W exactly.  Each o chunk is split once
// per CTA into bf16 hi / lo tiles in shared memory, from which every warp
// takes its A fragments by ldmatrix.
//
// Grid: (N / 256 column tiles) x (k splits) x (64-row blocks of M), about
// one CTA per SM.  A CTA of 4 warps streams its W[k range, 256 columns]
// (four 64-column TMA boxes per 64-deep k chunk, 128-byte swizzle) and
// o[64 rows, k range] through a 4-stage mbarrier ring; warp w owns columns
// 64 w .. 64 w + 63 over the whole k range, so no sums are exchanged and
// each o chunk is read once per 256 columns (the wider the tile, the fewer
// times the 4-byte o is re-read from L2 next to the 2-byte W).  Split
// partials go to the workspace and a second kernel adds them in fixed
// order (deterministic).  With programmatic dependent launch the W tiles of
// the first stages are requested before the attention's output is complete.
#include "pa_decode_mma.cuh"

namespace pa {
namespace {

constexpr int kWoThreads = 128;
constexpr int kWoWarps = 4;
constexpr int kWoBoxN = 64;    // columns per TMA box of W (128 bytes of bf16)
constexpr int kWoBoxes = 4;    // boxes per chunk: 256 columns per CTA
constexpr int kWoN = kWoBoxes * kWoBoxN;
constexpr int kWoWarpN = kWoN / kWoWarps;   // 64 columns (8 n8 tiles) per warp
constexpr int kWoK = 64;       // k per chunk: four k16 steps
constexpr int kWoStages = 4;
constexpr int kWoRows = 64;    // rows of o per CTA at most (4 m16 tiles)
constexpr int kWoBoxBytes = kWoK * kWoBoxN * 2;      // 8 KB
constexpr int kWoWBytes = kWoBoxes * kWoBoxBytes;    // 32 KB
// one 32-k fp32 box of o holds MT * 16 rows of 128 bytes
template <int MT>
struct WoGeo {
  static constexpr int ABox = MT * 16 * 128;
  static constexpr int Stage = kWoWBytes + 2 * ABox;   // multiple of 1024
  // the current chunk's o as bf16 hi and lo tiles [MT * 16 rows][64 k],
  // 128-byte rows with the 128-byte swizzle (conflict-free ldmatrix)
  static constexpr int XTile = MT * 16 * 128;
  static constexpr int Smem = kWoStages * Stage + 2 * XTile + 1024;
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

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

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

template <int MT>
__global__ void __launch_bounds__(kWoThreads) wo_kernel(const WoParams p,
                                                        const __grid_constant__ CUtensorMap tmW,
                                                        const __grid_constant__ CUtensorMap tmA) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t bars[kWoStages];
  __shared__ int s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nt = blockIdx.x % p.ntiles;
  const int s = (blockIdx.x / p.ntiles) % p.splits;
  const int mb = blockIdx.x / (p.ntiles * p.splits);
  using Gm = WoGeo<MT>;
  const int n0 = nt * kWoN, m0 = mb * kWoRows;
  const int c0 = s * p.chunks_per_split;
  const int nch = max(0, min(p.chunks_per_split, p.K / kWoK - c0));
  // the column tiles of a split read the same o chunks: start each at a
  // different chunk so that they do not all hit the same L2 lines at once
  const int rot = nch > 0 ? (nt * 5) % nch : 0;

  if (tid == 0) {
    for (int i = 0; i < kWoStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_fail = 0;
  }
  __syncthreads();
  const uint64_t pol = policy_evict_first();   // W: read once
  const uint64_t pol_o = policy_evict_last();   // o: read by every column tile
  auto chunk_k = [&](int c) { return (c0 + (c + rot) % nch) * kWoK; };
  auto issue_w = [&](int c) {   // thread 0: W rows of the c-th chunk, four boxes
    uint8_t *st = smem + (c % kWoStages) * Gm::Stage;
    mbar_arrive_expect_tx(&bars[c % kWoStages], Gm::Stage);
#pragma unroll
    for (int w = 0; w < kWoBoxes; ++w)
      tc::tma_rows(st + w * kWoBoxBytes, &tmW, n0 + w * kWoBoxN, chunk_k(c), &bars[c % kWoStages],
                   pol);
  };
  auto issue_a = [&](int c) {   // thread 0: o rows m0 .. m0 + 16 MT - 1, two 32-k boxes
    uint8_t *st = smem + (c % kWoStages) * Gm::Stage + kWoWBytes;
    const int k = chunk_k(c);
    tc::tma_rows(st, &tmA, k, m0, &bars[c % kWoStages], pol_o);
    tc::tma_rows(st + Gm::ABox, &tmA, k + 32, m0, &bars[c % kWoStages], pol_o);
  };
  const int pro = min(kWoStages, nch);
  if (tid == 0)
    for (int c = 0; c < pro; ++c) issue_w(c);   // W does not depend on the attention
  griddep_wait();                                // o of this call is complete
  if (tid == 0)
    for (int c = 0; c < pro; ++c) issue_a(c);

  // warp w: columns 64 w .. 64 w + 63 (8 n8 tiles), every k16 step
  float acc[MT][8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.f;

  // ldmatrix.trans row address: thread i -> matrix i / 8 = (k half, n half), row i % 8
  const int lm_k = ((lane >> 3) & 1) * 8 + (lane & 7);   // + 16 ks for k16 step ks
  const int lm_n = (lane >> 4) * 8;   // + 16 h for the h-th x4

  uint8_t *const xhi = smem + kWoStages * Gm::Stage, *const xlo = xhi + Gm::XTile;
  const uint32_t xhi_s = smem_u32(xhi), xlo_s = smem_u32(xlo);
  int issued = pro;
  for (int c = 0; c < nch; ++c) {
    const bool ok = mbar_wait(&bars[c % kWoStages], (c / kWoStages) & 1);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        set_err(p.hdr, PA_ERRF_WAIT_TIMEOUT);
        s_fail = 1;
      }
      break;
    }
    const uint8_t *st = smem + (c % kWoStages) * Gm::Stage;
    const uint32_t wbase = smem_u32(st) + warp * kWoBoxBytes;   // this warp's box
    const uint8_t *abase = st + kWoWBytes;
    // o of the chunk -> bf16 hi and lo tiles, each element once per CTA:
    // thread i takes 8 consecutive k of one row (one 16-byte piece of each tile)
    for (int i = tid; i < MT * 16 * 8; i += kWoThreads) {
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
    __syncthreads();   // the chunk's hi / lo tiles are complete
#pragma unroll
    for (int ks = 0; ks < kWoK / 16; ++ks) {
      const int kr = ks * 16 + lm_k;
      uint32_t b[4][4];   // four ldmatrix.x4: n8 tiles (2h, 2h + 1)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int n = lm_n + 16 * h;
        ldsm_x4_trans(wbase + kr * 128 + (((n >> 3) ^ (kr & 7)) << 4), b[h][0], b[h][1], b[h][2],
                      b[h][3]);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        // A fragments: matrix i = lanes 8i .. 8i + 7 -> rows (l & 7) + 8 ((l >> 3) & 1),
        // k chunk 2 ks + (l >> 4)
        const int ar = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int akc = 2 * ks + (lane >> 4);
        const uint32_t aoff = (uint32_t)(ar * 128 + ((akc ^ (ar & 7)) << 4));
        uint32_t ah[4], al[4];
        ldsm_x4(xhi_s + aoff, ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(xlo_s + aoff, al[0], al[1], al[2], al[3]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b0 = b[j >> 1][2 * (j & 1)], b1 = b[j >> 1][2 * (j & 1) + 1];
          mma_bf16(acc[mt][j], ah[0], ah[1], ah[2], ah[3], b0, b1);
          mma_bf16(acc[mt][j], al[0], al[1], al[2], al[3], b0, b1);
        }
      }
    }
    __syncthreads();   // stage consumed by every warp
    if (tid == 0 && issued < nch) {
      issue_w(issued);
      issue_a(issued);
      ++issued;
    }
  }
  if (s_fail) {   // only the last fill of each stage can still be in flight
    if (tid == 0)
      for (int c = max(issued - kWoStages, 0); c < issued; ++c)
        (void)mbar_wait(&bars[c % kWoStages], (c / kWoStages) & 1);
    return;
  }
  // ---- this warp's 64 columns, straight from the accumulators
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int m = m0 + mt * 16 + g + 8 * hh;
        const int n = n0 + warp * kWoWarpN + j * 8 + 2 * t;   // N is a multiple of 8: n + 1 < N too
        if (m >= p.M || n >= p.N) continue;
        const float v0 = acc[mt][j][2 * hh], v1 = acc[mt][j][2 * hh + 1];
        if (p.splits > 1)
          *reinterpret_cast<float2 *>(p.part + ((size_t)s * p.M + m) * p.N + n) = make_float2(v0, v1);
        else if (p.y_fp32)
          *reinterpret_cast<float2 *>(static_cast<float *>(p.y) + (size_t)m * p.N + n) =
              make_float2(v0, v1);
        else
          *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.y) + (size_t)m * p.N + n) =
              __floats2bfloat162_rn(v0, v1);
      }
}

// y = sum over splits of the partials, in split order
__global__ void wo_reduce_kernel(const WoParams p) {
  griddep_wait();
  const size_t total = (size_t)p.M * p.N;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
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
  const unsigned rgrid = (unsigned)std::min<size_t>((total + 255) / 256, 2048);
  return launch_pdl(wo_reduce_kernel, rgrid, 256, 0, s, p);
}

}  // namespace pa
