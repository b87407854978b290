// pa_sparse.cu -- block-sparse decode by per-block mean keys ("vLLM-SM70",
// "Known limitations" and its production fixes: sparse-decode selection
// over per-block mean keys, blocks of 64 tokens, at most 4096 of them; mean
// keys refreshed for every request of a decode batch).
//
//   means_kernel   mean dequantised key of sparse blocks [first[b], nsb(b))
//                  of every sequence: one CTA per (sequence, block, kv head)
//   score_kernel   score[b, h, j] = max over the query heads g of kv head h
//                  of q_g . mean_j: one lane per (sequence, kv head, block)
//   select_kernel  one CTA per (sequence, kv head): the top_k scores (ties to
//                  the lower index) by a bitwise search for the n-th largest
//                  (score, index) key, then the selected blocks in ascending
//                  order written as a block table of a per-kv-head virtual
//                  sequence: logical block lb of the sequence becomes entry
//                  table[b][lb] * Hkv + h, which is the id of that (block,
//                  kv head) tile in the pool viewed as [NB * Hkv, 1, 16, D].
// The attention itself is the ordinary decode over that view (B * Hkv
// sequences of one kv head and G query heads each): only the work list
// changes.  Only the sequence's last sparse block can be partial, and it
// sorts last, so every virtual sequence is whole 16-token blocks but its
// last.
#include <algorithm>
#include <atomic>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kSelThreads = 256;

// dequantised key elements d0 .. d0 + 7 of pool row `row` (fp32, exactly the
// values the attention kernels use)
__device__ __forceinline__ void key8(const KvView &kv, size_t row, int d0, float (&f)[8]) {
  const int D = kv.D;
  if (kv.dtype == PA_KV_BF16) {
    const uint4 u = *reinterpret_cast<const uint4 *>(
        reinterpret_cast<const __nv_bfloat16 *>(kv.k) + row * D + d0);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = bf16x2_to_f2(w[j]);
      f[2 * j] = x.x;
      f[2 * j + 1] = x.y;
    }
  } else if (kv.dtype == PA_KV_INT8) {
    const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const int8_t *>(kv.k) +
                                                     row * D + d0);
    s8x4_to_f4(u.x, f);
    s8x4_to_f4(u.y, f + 4);
    const float s = fp16_bits_to_f(reinterpret_cast<const uint16_t *>(kv.ks)[row]);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = f[j] * s;
  } else if (kv.dtype == PA_KV_FP8) {
    const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(kv.k) +
                                                     row * D + d0);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = h2u_to_f2(e4m3x2_u16_to_h2(w[j >> 1] >> (16 * (j & 1))));
      f[2 * j] = x.x * kv.kg;
      f[2 * j + 1] = x.y * kv.kg;
    }
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(
        reinterpret_cast<const uint8_t *>(kv.k) + row * (D / 2) + d0 / 2);
    const uint32_t s2 =
        e4m3_to_h2_dup(reinterpret_cast<const uint8_t *>(kv.ks)[row * (D / 16) + d0 / 16]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = h2u_to_f2(hmul2_u32(e2m1x2_to_h2((u >> (8 * j)) & 0xffu), s2));
      f[2 * j] = x.x * kv.kg;
      f[2 * j + 1] = x.y * kv.kg;
    }
  }
}

__device__ __forceinline__ int seq_len_of(const int *seq_lens, int b, int capacity) {
  const int L = seq_lens[b];
  return L < 0 ? 0 : (L > capacity ? capacity : L);
}

// one CTA per (b, j, h); warp w sums the 16-token block j * sb / 16 + w with
// its 16 row loads in flight, then the warps' sums are added in fixed order
__global__ void __launch_bounds__(512) means_kernel(const KvView kv, const int *tables, int stride,
                                                    const int *seq_lens, const int *first, int count,
                                                    int B, int sb, int max_nsb, float *means,
                                                    uint32_t *hdr) {
  __shared__ float part[16][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;   // sb / 16
  const int H = kv.hkv, D = kv.D;
  const int h = (int)(blockIdx.x % H);
  const int b = (int)(blockIdx.x / ((unsigned)H * count));
  const int j = (first ? max(first[b], 0) : 0) + (int)((blockIdx.x / H) % count);
  const int L = seq_len_of(seq_lens, b, stride * kBlock);
  const int lo = j * sb, hi = min(L, lo + sb);
  if (lo >= hi || j >= max_nsb) return;   // uniform over the CTA
  const int d0 = lane * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int t0 = lo + warp * kBlock;
  if (t0 < hi) {
    const int phys = tables[(size_t)b * stride + t0 / kBlock];
    if (phys < 0 || phys >= kv.num_blocks) {   // skipped like the attention kernels do
      if (lane == 0) set_err(hdr, PA_ERRF_BAD_BLOCK_ID);
    } else if (d0 < D) {
      const int n = min(kBlock, hi - t0);
      const size_t row0 = ((size_t)phys * H + h) * kBlock;
#pragma unroll
      for (int t = 0; t < kBlock; ++t) {
        if (t < n) {
          float f[8];
          key8(kv, row0 + t, d0, f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
      }
    }
  }
  if (d0 < D) {
#pragma unroll
    for (int i = 0; i < 8; ++i) part[warp][d0 + i] = acc[i];
  }
  __syncthreads();
  const float inv = __frcp_rn((float)(hi - lo));
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float sum = 0.f;
    for (int w = 0; w < nw; ++w) sum += part[w][d];
    means[(((size_t)b * max_nsb + j) * H + h) * D + d] = sum * inv;
  }
}

// Eight lanes per sparse block, two blocks per lane group: a CTA of 128
// threads scores a run of consecutive blocks of one (b, h), 32 per step of
// its four warps; the runs are as long as makes the grid one round of the
// GPU's resident CTAs.  Lane l8 of a group reads float4 l8, l8 + 8, ... of its two blocks'
// mean rows, so the four groups of a load instruction read four whole
// 128-byte lines (coalesced); every query float4 read from shared memory
// serves both blocks, and the eight partial dots of each head are added by
// three shuffles.  The mean rows are read with the streaming (evict-first)
// cache hint: they are read once per step and would otherwise push out of L2
// what the kernels after them reuse (decode step 0.154 -> 0.142 ms at
// 8 x 262K).
constexpr int kScoreThreads = 128;

// per_cta: blocks per CTA, a multiple of 8 (a warp step's blocks)
template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(
    const __nv_bfloat16 *q, int Hq, const int *seq_lens, int capacity, int B, int H, int D,
    int sb, int max_nsb, int per_cta, const float *means, float *scores) {
  __shared__ float4 sq[G][256 / 4];
  const int chunks = (max_nsb + per_cta - 1) / per_cta;
  const int c = blockIdx.x % chunks;
  const int h = (blockIdx.x / chunks) % H;
  const int b = blockIdx.x / (chunks * H);
  for (int i = threadIdx.x; i < G * D / 4; i += kScoreThreads) {
    const int g = i / (D / 4), d4 = i % (D / 4);
    const uint2 u = *reinterpret_cast<const uint2 *>(q + ((size_t)b * Hq + h * G + g) * D + 4 * d4);
    const float2 lo = bf16x2_to_f2(u.x), hi = bf16x2_to_f2(u.y);
    sq[g][d4] = make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  __syncthreads();
  const int L = seq_len_of(seq_lens, b, capacity);
  // blocks beyond the means' capacity have no mean (the selection flags them)
  const int nsb = min((L + sb - 1) / sb, max_nsb);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> 3, l8 = lane & 7;
  const int per = D / 32;   // float4 of a row per lane
  const int j_end = min(max_nsb, (c + 1) * per_cta);
  for (int step = 0; step * 32 < per_cta; ++step) {
    const int j0 = c * per_cta + step * 32 + warp * 8;   // the warp's first block
    if (j0 >= j_end) break;                              // the whole warp
    const int ja = j0 + sub, jb = ja + 4;                   // this group's two blocks
    float acc[2][G];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) acc[u][g] = 0.f;
    float4 x[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = u ? jb : ja;
      const float4 *m = reinterpret_cast<const float4 *>(means + (((size_t)b * max_nsb + j) * H + h) * D);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[u][i] = (i < per && j < nsb) ? __ldcs(&m[l8 + 8 * i]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < per) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 y = sq[g][l8 + 8 * i];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            acc[u][g] = fmaf(x[u][i].x, y.x, fmaf(x[u][i].y, y.y,
                        fmaf(x[u][i].z, y.z, fmaf(x[u][i].w, y.w, acc[u][g]))));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = u ? jb : ja;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        acc[u][g] += __shfl_xor_sync(0xffffffffu, acc[u][g], 1);
        acc[u][g] += __shfl_xor_sync(0xffffffffu, acc[u][g], 2);
        acc[u][g] += __shfl_xor_sync(0xffffffffu, acc[u][g], 4);
      }
      float sc = kNegInf;
      if (j < nsb) {
#pragma unroll
        for (int g = 0; g < G; ++g) sc = fmaxf(sc, acc[u][g]);
      }
      if (l8 == 0 && j < max_nsb) scores[((size_t)b * H + h) * max_nsb + j] = sc;
    }
  }
}

// (score, index) -> key ordered like (score descending, index ascending)
__device__ __forceinline__ unsigned long long sel_key(float s, int j) {
  uint32_t u = __float_as_uint(s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // order-preserving for finite and -inf
  return ((unsigned long long)u << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)j);
}

// One CTA of 256 threads per (b, h), each thread holding up to 16
// (score, index) keys in registers as two words (score key, index key).
// The keys are unique, so the top n are exactly the keys >= the n-th
// largest, which is found bit by bit from the top: keep a bit when at least
// n keys are >= the prefix with it set (warp ballots, per-warp counts in
// shared memory, one barrier per bit).  The bits above the highest one in
// which the valid score words differ are common to all of them and are not
// searched (one AND / OR reduction first), and the search stops as soon as
// exactly n keys reach the prefix.  While the score word is searched the
// prefix's index word is 0, so comparing score words alone gives the same
// counts; when exactly n keys reach the score prefix (no tie at the
// boundary) it is the answer and the index word is not searched.  Index
// bits 31..12 are 1 in every key (index < 4096) and are not searched.
// A bitmap of the winners gives each one its rank in ascending block order;
// the winners' block-table entries are then gathered with all of a thread's
// loads in flight before its stores.
__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const int *tables, int stride, const int *seq_lens, int B, int H, int sb, int max_nsb,
    int top_k, const float *scores, int *selected, int *vtables, int vstride, int *vlens,
    int num_blocks, uint32_t *err) {
  constexpr int kPer = 4096 / kSelThreads;   // keys per thread
  constexpr int kWarpsSel = kSelThreads / 32;
  constexpr int kGather = 8;                 // table entries in flight per thread
  __shared__ uint32_t s_flag[4096 / 32], s_wpre[4096 / 32];
  __shared__ int s_cnt[2][kWarpsSel];
  __shared__ uint32_t s_and[kWarpsSel], s_or[kWarpsSel];
  __shared__ int s_rank[4096];               // rank -> sparse block index
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = seq_len_of(seq_lens, b, stride * kBlock);
  if (tid == 0) {
    const int raw = seq_lens[b];
    if (raw < 0) atomicOr(err, PA_ERRF_NEG_LEN);
    if (raw > stride * kBlock) atomicOr(err, PA_ERRF_LEN_OVER_CAPACITY);
  }
  int nsb = (L + sb - 1) / sb;
  if (nsb > max_nsb) {   // beyond the means' capacity: attended over its first blocks only
    if (tid == 0) atomicOr(err, PA_ERRF_PLAN_OVERFLOW);
    nsb = max_nsb;
    L = nsb * sb;
  }
  const int n = min(top_k, nsb);
  const float *sc = scores + ((size_t)b * H + h) * max_nsb;
  // the score row is read up to max_nsb whatever the length (in flight
  // together with the length)
  float sv[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = tid + i * kSelThreads;
    sv[i] = j < max_nsb ? sc[j] : 0.f;
  }
  uint32_t khi[kPer], klo[kPer];   // score word, index word; 0 / 0 is below every real key
  uint32_t kand = 0xFFFFFFFFu, kor = 0u;   // over this thread's valid score words
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = tid + i * kSelThreads;
    const unsigned long long k = j < nsb ? sel_key(sv[i], j) : 0ull;
    khi[i] = (uint32_t)(k >> 32);
    klo[i] = (uint32_t)k;
    if (j < nsb) {
      kand &= khi[i];
      kor |= khi[i];
    }
  }
  for (int i = tid; i < 4096 / 32; i += kSelThreads) s_flag[i] = 0;
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  if (lane == 0) {
    s_and[warp] = kand;
    s_or[warp] = kor;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarpsSel; ++w) {
    kand &= s_and[w];
    kor |= s_or[w];
  }
  // the n-th largest key (n < nsb), else 0 / 0 = take all
  uint32_t thr_hi = 0, thr_lo = 0;
  int buf = 0;
  // keys of the whole CTA for which ge(i) holds (one barrier; the next call
  // writes the other buffer, so no second barrier is needed)
  auto count_ge = [&](auto ge) {
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) cnt += __popc(__ballot_sync(0xffffffffu, ge(i)));
    if (lane == 0) s_cnt[buf][warp] = cnt;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < kWarpsSel; ++w) tot += s_cnt[buf][w];
    buf ^= 1;
    return tot;
  };
  if (n < nsb) {
    // every valid score word has the bits above `top` of kand; every key
    // that is not valid is 0 and below them all
    const uint32_t diff = kand ^ kor;
    const int top = diff ? 31 - __clz(diff) : -1;
    thr_hi = top < 0 ? kand : top < 31 ? (kand & ~((2u << top) - 1u)) : 0u;
    bool exact = false;   // exactly n keys reach thr_hi
    for (int bit = top; bit >= 0 && !exact; --bit) {   // the score word
      const uint32_t cand = thr_hi | (1u << bit);
      const int c = count_ge([&](int i) { return khi[i] >= cand; });
      if (c >= n) {
        thr_hi = cand;
        exact = c == n;
      }
    }
    if (!exact && count_ge([&](int i) { return khi[i] >= thr_hi; }) != n) {   // a tie at the boundary
      thr_lo = 0xFFFFF000u;
      for (int bit = 11; bit >= 0; --bit) {   // the index word
        const uint32_t cand = thr_lo | (1u << bit);
        if (count_ge([&](int i) { return khi[i] > thr_hi || (khi[i] == thr_hi && klo[i] >= cand); }) >= n)
          thr_lo = cand;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = tid + i * kSelThreads;
    if (j < nsb && (khi[i] > thr_hi || (khi[i] == thr_hi && klo[i] >= thr_lo)))
      atomicOr(&s_flag[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  if (warp == 0) {   // exclusive prefix of the bitmap's word counts
    uint32_t run = 0;
    for (int base = 0; base < 4096 / 32; base += 32) {
      const uint32_t c = __popc(s_flag[base + lane]);
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      s_wpre[base + lane] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  const size_t vrow = (size_t)b * H + h;
  for (int j = tid; j < nsb; j += kSelThreads) {
    const uint32_t w = s_flag[j >> 5];
    if (!((w >> (j & 31)) & 1u)) continue;
    const int r = (int)(s_wpre[j >> 5] + __popc(w & ((1u << (j & 31)) - 1u)));
    s_rank[r] = j;
    if (selected) selected[vrow * top_k + r] = j;
  }
  __syncthreads();
  // block-table entries of the winners: entry (r, i) = 16-token block i of
  // the rank-r winner; all of a thread's loads are issued before its stores
  const int bps = sb / kBlock;   // 16-token blocks per sparse block
  const int nblk = (L + kBlock - 1) / kBlock;
  const int total = n * bps;
  const int *trow = tables + (size_t)b * stride;
  int *vrow_t = vtables + vrow * vstride;
  for (int e0 = 0; e0 < total; e0 += kGather * kSelThreads) {
    int phys[kGather];
    bool have[kGather];   // an entry of a block inside the sequence
#pragma unroll
    for (int k = 0; k < kGather; ++k) {
      const int e = e0 + k * kSelThreads + tid;
      const int lb = e < total ? s_rank[e / bps] * bps + e % bps : nblk;
      have[k] = lb < nblk;
      phys[k] = have[k] ? trow[lb] : 0;
    }
#pragma unroll
    for (int k = 0; k < kGather; ++k) {
      const int e = e0 + k * kSelThreads + tid;
      if (have[k]) vrow_t[e] = (phys[k] >= 0 && phys[k] < num_blocks) ? phys[k] * H + h : -1;
    }
  }
  if (selected)
    for (int i = n + tid; i < top_k; i += kSelThreads) selected[vrow * top_k + i] = -1;
  if (tid == 0) {
    // keys of the selected blocks: whole sparse blocks, the sequence's last
    // one (if chosen) only up to L
    const int last = nsb - 1;
    const bool last_in = nsb > 0 && ((s_flag[last >> 5] >> (last & 31)) & 1u);
    vlens[vrow] = last_in ? (n - 1) * sb + (L - last * sb) : n * sb;
  }
}

}  // namespace

cudaError_t launch_means(const KvView &kv, const int *tables, int stride, const int *seq_lens,
                         const int *first, int count, int B, int sb, int max_nsb, float *means,
                         uint32_t *hdr, cudaStream_t s) {
  const long long grid = (long long)B * count * kv.hkv;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  means_kernel<<<(unsigned)grid, 32 * (sb / kBlock), 0, s>>>(kv, tables, stride, seq_lens, first,
                                                             count, B, sb, max_nsb, means, hdr);
  return cudaGetLastError();
}

// CTAs of score_kernel<G> resident on the whole GPU (SMs x CTAs per SM), 0
// if unknown; asked once per (device, G)
template <int G>
static int score_occupancy() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_kernel<G>, kScoreThreads, 0) !=
      cudaSuccess)
    return 0;
  return n;
}

static int score_slots(int G) {
  constexpr int kDevs = 16;
  static std::atomic<int> known[kDevs][9];   // slots + 1, 0 = not yet asked
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || G < 1 || G > 8) return 0;
  std::atomic<int> *slot = dev >= 0 && dev < kDevs ? &known[dev][G] : nullptr;
  if (slot) {
    const int v = slot->load(std::memory_order_relaxed);
    if (v > 0) return v - 1;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  int occ = 0;
  switch (G) {
    case 1: occ = score_occupancy<1>(); break;
    case 2: occ = score_occupancy<2>(); break;
    case 3: occ = score_occupancy<3>(); break;
    case 4: occ = score_occupancy<4>(); break;
    case 5: occ = score_occupancy<5>(); break;
    case 6: occ = score_occupancy<6>(); break;
    case 7: occ = score_occupancy<7>(); break;
    case 8: occ = score_occupancy<8>(); break;
  }
  const int n = occ * sms;
  if (slot && n > 0) slot->store(n + 1, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_sparse_select(const KvView &kv, const __nv_bfloat16 *q, int Hq,
                                 const int *tables, int stride, const int *seq_lens, int B, int sb,
                                 int max_nsb, int top_k, const float *means, float *scores,
                                 int *selected, int *vtables, int vstride, int *vlens,
                                 uint32_t *err, cudaStream_t s) {
  const int H = kv.hkv, G = Hq / H;
  if (G < 1 || G > 8) return cudaErrorInvalidValue;
  // one round of resident CTAs: the (b, h) rows' blocks are cut into as many
  // chunks as fill the GPU's resident CTAs once (the last of two rounds was
  // a third full with 128 blocks per CTA: 30.7 us for 8 x 4 x 4096 blocks)
  const long long rows = (long long)B * H;
  const int slots = score_slots(G);
  const long long cpr = slots > 0 ? std::max(1LL, slots / rows) : 1LL;
  int per_cta = (int)((max_nsb + cpr - 1) / cpr);
  per_cta = std::max(8, (per_cta + 7) / 8 * 8);
  const long long grid = rows * ((max_nsb + per_cta - 1) / per_cta);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int cap = stride * kBlock;
#define PA_SCORE_CASE(GG)                                                                    \
  case GG:                                                                                   \
    score_kernel<GG><<<(unsigned)grid, kScoreThreads, 0, s>>>(q, Hq, seq_lens, cap, B, H,    \
                                                              kv.D, sb, max_nsb, per_cta,    \
                                                              means, scores);                \
    break;
  switch (G) {
    PA_SCORE_CASE(1) PA_SCORE_CASE(2) PA_SCORE_CASE(3) PA_SCORE_CASE(4)
    PA_SCORE_CASE(5) PA_SCORE_CASE(6) PA_SCORE_CASE(7) PA_SCORE_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef PA_SCORE_CASE
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  select_kernel<<<B * H, kSelThreads, 0, s>>>(tables, stride, seq_lens, B, H, sb, max_nsb, top_k,
                                                  scores, selected, vtables, vstride, vlens,
                                                  kv.num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pa
