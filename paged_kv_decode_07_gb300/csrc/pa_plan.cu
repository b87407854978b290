// pa_plan.cu -- device-side split-K planner.
//
// Splits every sequence's keys into partitions of whole 16-token blocks so
// that partitions of all sequences run in parallel across the SMs
// (flash-decoding; "split-KV merge", "vLLM Fork with focus on GB10
// Homelabs", "Acknowledgments").  Like stream-K scheduling ("SM120 Stream-K
// Decode Optimization" on the same page), the K dimension of a small-M
// problem is what gets spread across SMs; here it is the key axis.
//
// One CTA of 1024 threads reads seq_lens on the device (no host read, so a
// call can be captured in a CUDA graph) and writes:
//   units[u]  = {parts, slot_base, nblk, len}
//   items[j]  = {unit, kvh, blk_begin, blk_end, part, parts, slot}
// Partition size W (blocks) = max(min_split, ceil(total_blocks * Hkv /
// target_items)) unless fixed by the caller; when every sequence has the
// same length, W then grows until the item count is a whole number of
// rounds of the attention kernel's resident CTAs (the number of rounds from
// a cost model: a round costs its items' blocks plus a fixed cost per item).  parts_u = ceil(nblk_u /
// W); blocks are split evenly, ceil(nblk_u / parts_u) per part (never
// empty).
// Items of multi-part units come first (they are about W blocks each), then
// the single-part ones (shorter), a longest-first order for the hardware's
// in-order CTA dispatch.
#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kThreads = 1024;
// batches of up to this many sequences keep the planner's per-sequence
// arrays in shared memory (the item sweep's binary searches then cost no
// global-memory round trips); larger ones use the workspace scratch
constexpr int kSmemGroups = 2048;

// A group is one sequence: in virtual mode with q_len > 1 its q_len units
// share partition boundaries (taken from the group's longest unit), and its
// items are ordered (part, query row, kv head) so the q_len reads of the
// same key blocks run back to back and hit L2.
__device__ __forceinline__ int group_size(const PlanParams &p) {
  return p.virt == 1 ? p.Q : (p.virt == 2 ? p.RG : 1);
}

__device__ __forceinline__ int unit_len(const PlanParams &p, int u, uint32_t &err) {
  const int b = u / group_size(p);
  const int i = p.virt == 1 ? u % p.Q : p.Q - 1;   // row groups see up to the last query
  int L = p.seq_lens[b];
  if (L < 0) {
    err |= PA_ERRF_NEG_LEN;
    L = 0;
  }
  if (L > p.capacity) {
    err |= PA_ERRF_LEN_OVER_CAPACITY;
    L = p.capacity;
  }
  if (L > 0 && L < p.Q) err |= PA_ERRF_LEN_LT_QLEN;
  if (L == 0) return 0;
  int n = L - p.Q + 1 + i;  // keys visible to the unit's last row
  return n > 0 ? n : 0;
}

// exclusive block-wide scan of a pair of ints; returns totals in tot
__device__ __forceinline__ int2 block_scan2(int2 v, int2 &tot) {
  __shared__ int2 warp_sums[kThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int a = __shfl_up_sync(0xffffffffu, x.x, o);
    int b = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) {
      x.x += a;
      x.y += b;
    }
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int2 s = warp_sums[lane];
    int2 y = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int a = __shfl_up_sync(0xffffffffu, y.x, o);
      int b = __shfl_up_sync(0xffffffffu, y.y, o);
      if (lane >= o) {
        y.x += a;
        y.y += b;
      }
    }
    warp_sums[lane] = make_int2(y.x - s.x, y.y - s.y);  // exclusive warp offsets
    if (lane == 31) tot = y;                             // only thread 31 of warp 0 sets it
  }
  __syncthreads();
  int2 off = warp_sums[w];
  int2 r = make_int2(off.x + x.x - v.x, off.y + x.y - v.y);
  __syncthreads();
  return r;
}

template <typename P>
__device__ __forceinline__ int upper_bound_minus1(const P *pre, int n, int j) {
  int lo = 0, hi = n;  // first index with pre[idx] > j
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (pre[mid] > j)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo - 1;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(PlanParams p) {
  __shared__ unsigned long long s_total;
  __shared__ uint32_t s_err;
  __shared__ int2 s_tot;
  __shared__ int s_W, s_round;
  __shared__ int s_gmin, s_gmax;   // least / most blocks of a group's partition basis
  __shared__ int s_pa[kSmemGroups], s_pb[kSmemGroups];         // item prefix per group
  __shared__ int s_parts[kSmemGroups], s_nblk[kSmemGroups], s_slot[kSmemGroups];
  griddep_launch();   // the attention kernel may launch now; it waits for this grid to finish
  const int tid = threadIdx.x;
  const int U = p.B * group_size(p);
  if (tid == 0) {
    s_total = 0;
    s_err = 0;
    s_round = 0;
    s_gmin = 0x7fffffff;
    s_gmax = 0;
  }
  __syncthreads();

  const int GS = group_size(p);
  const int NG = p.B;                    // groups = sequences
  const bool sm = NG <= kSmemGroups;
  int *pa = sm ? s_pa : p.prefix_a;
  int *pb = sm ? s_pb : p.prefix_b;
  // sweep 1: total key blocks over all units (the work the kernel streams)
  uint32_t err = 0;
  unsigned long long tot = 0;
  for (int u = tid; u < U; u += kThreads) {
    int n = unit_len(p, u, err);
    tot += (unsigned long long)((n + kBlock - 1) / kBlock);
  }
  // the blocks every group partitions (those of its longest unit): the same
  // in every group when the sequences have equal lengths
  int gmin = 0x7fffffff, gmax = 0;
  if (p.resident > 0 && p.split_blocks <= 0) {
    uint32_t e1 = 0;
    for (int g = tid; g < NG; g += kThreads) {
      int nmax = 0;
      for (int i = 0; i < GS; ++i) nmax = max(nmax, unit_len(p, g * GS + i, e1));
      const int nb = (nmax + kBlock - 1) / kBlock;
      gmin = min(gmin, nb);
      gmax = max(gmax, nb);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_down_sync(0xffffffffu, tot, o);
    gmin = min(gmin, __shfl_down_sync(0xffffffffu, gmin, o));
    gmax = max(gmax, __shfl_down_sync(0xffffffffu, gmax, o));
  }
  if ((tid & 31) == 0) {
    atomicAdd(&s_total, tot);
    atomicMin(&s_gmin, gmin);
    atomicMax(&s_gmax, gmax);
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();
  if (tid == 0) {
    long long W;
    if (p.split_blocks > 0) {
      W = p.split_blocks;
    } else {
      long long work = (long long)s_total * p.hkv;
      W = (work + p.target_items - 1) / p.target_items;
      if (W < p.min_split_blocks) W = p.min_split_blocks;
      // Equal-length groups give items of one size, and the kernel then takes
      // as long as the rounds of resident CTAs its items fill: a last round
      // that is only partly full costs a whole round, and every item adds a
      // fixed cost.  Over k = 1 .. the rounds the target's item count fills
      // completely, with parts_k = the most partitions per unit that fit k
      // rounds, the partitions take the k of least k * (nb / parts_k + c).
      const int nb = s_gmax;
      if (p.resident > 0 && nb > 0 && s_gmin == nb) {
        const long long per = (long long)NG * GS * p.hkv;   // items per partition index
        const long long items0 = per * ((nb + W - 1) / W);
        // at most 64 rounds are weighed: past that a partial round costs
        // under 2 % (and thread 0 stays quick for very large batches)
        const long long kmax = min(items0 / p.resident, 64LL);
        long long best_w = 0, best_t = 0;
        for (long long k = 1; k <= kmax; ++k) {
          const long long parts = k * p.resident / per;
          if (parts < 1) continue;
          const long long wk = (nb + parts - 1) / parts;
          const long long t = k * (wk + p.item_cost);
          if (best_w == 0 || t < best_t) {
            best_w = wk;
            best_t = t;
          }
        }
        if (best_w > 0) {
          W = max(W, best_w);
          s_round = p.resident;
        }
      }
    }
    if (W < 1) W = 1;
    if (W > (1 << 30)) W = 1 << 30;
    s_W = (int)W;
  }
  __syncthreads();
  const int W = s_W;

  // sweep 2: per group, partitions from its longest unit; multi-part groups
  // get items and slots first, single-part groups after
  int2 carry = make_int2(0, 0);
  for (int base = 0; base < NG; base += kThreads) {
    const int g = base + tid;
    uint32_t e2 = 0;
    int nmax = 0;
    if (g < NG)
      for (int i = 0; i < GS; ++i) nmax = max(nmax, unit_len(p, g * GS + i, e2));
    const int nblk = (nmax + kBlock - 1) / kBlock;
    const int parts = nblk ? (nblk + W - 1) / W : 0;
    const int multi = parts > 1;
    int2 v = make_int2(multi ? parts * GS * p.hkv : 0, multi ? parts * GS : 0);
    int2 ex = block_scan2(v, s_tot);
    if (g < NG) {
      pa[g] = carry.x + ex.x;
      if (sm) {
        s_parts[g] = parts;
        s_nblk[g] = nblk;
        s_slot[g] = multi ? carry.y + ex.y : -1;
      }
      for (int i = 0; i < GS; ++i) {
        UnitInfo ui;
        ui.parts = parts;
        ui.slot_base = multi ? carry.y + ex.y + i * parts : -1;
        ui.nblk = nblk;
        ui.len = unit_len(p, g * GS + i, e2);
        p.units[g * GS + i] = ui;
      }
    }
    __syncthreads();
    carry.x += s_tot.x;
    carry.y += s_tot.y;
    __syncthreads();
  }
  const int items_a = carry.x, slots = carry.y;
  int2 carry_b = make_int2(0, 0);
  for (int base = 0; base < NG; base += kThreads) {
    const int g = base + tid;
    int single = 0;
    if (g < NG) single = (sm ? s_parts[g] : p.units[g * GS].parts) == 1;
    int2 v = make_int2(single ? GS * p.hkv : 0, 0);
    int2 ex = block_scan2(v, s_tot);
    if (g < NG) pb[g] = carry_b.x + ex.x;
    __syncthreads();
    carry_b.x += s_tot.x;
    __syncthreads();
  }
  int num_items = items_a + carry_b.x;
  if (num_items > p.max_items || slots > p.max_slots) {
    // cannot happen for a workspace sized by pa_workspace_bytes; never write
    // past the buffers
    num_items = 0;
    if (tid == 0) atomicOr(&s_err, PA_ERRF_PLAN_OVERFLOW);
  }
  __syncthreads();

  // sweep 3: write the items, (part, query row, kv head) within a group
  const int per_part = GS * p.hkv;
  for (int j = tid; j < num_items; j += kThreads) {
    int g, local;
    if (j < items_a) {
      g = upper_bound_minus1(pa, NG, j);
      local = j - pa[g];
    } else {
      g = upper_bound_minus1(pb, NG, j - items_a);
      local = j - items_a - pb[g];
    }
    const int part = local / per_part, rem = local % per_part;
    const int i = rem / p.hkv, kvh = rem % p.hkv;
    const int u = g * GS + i;
    int parts, nblk, slot_base;
    if (sm) {   // every unit of a group shares its parts and blocks
      parts = s_parts[g];
      nblk = s_nblk[g];
      slot_base = parts > 1 ? s_slot[g] + i * parts : -1;
    } else {
      const UnitInfo ui = p.units[u];
      parts = ui.parts;
      nblk = ui.nblk;
      slot_base = ui.slot_base;
    }
    const int chunk = (nblk + parts - 1) / parts;
    WorkItem it;
    it.unit = u;
    it.kvh = kvh;
    it.blk_begin = part * chunk;
    it.blk_end = min(nblk, it.blk_begin + chunk);
    it.part = part;
    it.parts = parts;
    it.slot = parts > 1 ? slot_base + part : -1;
    it.pad = 0;
    p.items[j] = it;
  }
  if (tid == 0) {
    p.hdr[HDR_ERR] = s_err | (p.extra_err ? *p.extra_err : 0u);
    p.hdr[HDR_NUM_ITEMS] = (uint32_t)num_items;
    p.hdr[HDR_SPLIT] = (uint32_t)W;
    p.hdr[HDR_NUM_SLOTS] = (uint32_t)slots;
    p.hdr[HDR_ROUND] = (uint32_t)s_round;
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams &pp, cudaStream_t s) {
  plan_kernel<<<1, kThreads, 0, s>>>(pp);
  return cudaGetLastError();
}

}  // namespace pa
