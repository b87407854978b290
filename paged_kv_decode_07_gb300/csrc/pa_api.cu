// pa_api.cu -- host side of the C ABI declared in include/pa.h: argument
// validation (errors return before anything is launched), workspace layout,
// and the planner -> attention kernel -> merge launch sequence.
#include <atomic>
#include <cmath>
#include <cstring>

#include "pa_launch.h"

namespace pa {
cudaError_t launch_decode_simt_bf16(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_simt_int8(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_simt_nvfp4(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_simt_fp8(const AttnParams &p, int grid, cudaStream_t s);

cudaError_t launch_decode_tc_bf16(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_tc_int8(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_tc_nvfp4(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_decode_tc_fp8(const AttnParams &p, int grid, cudaStream_t s);

cudaError_t launch_decode_tc_cluster_bf16(const AttnParams &p, int P, cudaStream_t s);
cudaError_t launch_decode_tc_cluster_int8(const AttnParams &p, int P, cudaStream_t s);
cudaError_t launch_decode_tc_cluster_nvfp4(const AttnParams &p, int P, cudaStream_t s);
cudaError_t launch_decode_tc_cluster_fp8(const AttnParams &p, int P, cudaStream_t s);

// the single-launch decode: one thread-block cluster of P CTAs per
// (sequence, kv head), partials merged in distributed shared memory
cudaError_t launch_decode_tc_cluster(const AttnParams &p, int P, cudaStream_t s) {
  switch (p.kv.dtype) {
    case PA_KV_BF16: return launch_decode_tc_cluster_bf16(p, P, s);
    case PA_KV_INT8: return launch_decode_tc_cluster_int8(p, P, s);
    case PA_KV_NVFP4: return launch_decode_tc_cluster_nvfp4(p, P, s);
    case PA_KV_FP8: return launch_decode_tc_cluster_fp8(p, P, s);
  }
  return cudaErrorInvalidValue;
}

int decode_tc_occupancy_bf16(int D, int R);
int decode_tc_occupancy_int8(int D, int R);
int decode_tc_occupancy_nvfp4(int D, int R);
int decode_tc_occupancy_fp8(int D, int R);

// CTAs of the tensor-core decode kernel one SM holds at once, 0 if unknown;
// queried once per (device, format, head dim, rows) and kept
int decode_tc_occupancy(int dtype, int D, int R) {
  constexpr int kDevs = 16;
  static std::atomic<int> known[kDevs][4][2][kMaxG + 1];   // occupancy + 1, 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dtype < PA_KV_BF16 || dtype > PA_KV_FP8 || R < 1 || R > kMaxG || (D != 128 && D != 256))
    return 0;
  std::atomic<int> *slot = dev >= 0 && dev < kDevs ? &known[dev][dtype][D == 256][R] : nullptr;
  if (slot) {
    const int v = slot->load(std::memory_order_relaxed);
    if (v > 0) return v - 1;
  }
  int n = 0;
  switch (dtype) {
    case PA_KV_BF16: n = decode_tc_occupancy_bf16(D, R); break;
    case PA_KV_INT8: n = decode_tc_occupancy_int8(D, R); break;
    case PA_KV_NVFP4: n = decode_tc_occupancy_nvfp4(D, R); break;
    case PA_KV_FP8: n = decode_tc_occupancy_fp8(D, R); break;
  }
  if (slot && n > 0) slot->store(n + 1, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_decode_tc(const AttnParams &p, int grid, cudaStream_t s) {
  switch (p.kv.dtype) {
    case PA_KV_BF16: return launch_decode_tc_bf16(p, grid, s);
    case PA_KV_INT8: return launch_decode_tc_int8(p, grid, s);
    case PA_KV_NVFP4: return launch_decode_tc_nvfp4(p, grid, s);
    case PA_KV_FP8: return launch_decode_tc_fp8(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

int tc_supported(int dtype, int D, int R) {
  return (dtype == PA_KV_BF16 || dtype == PA_KV_INT8 || dtype == PA_KV_NVFP4 || dtype == PA_KV_FP8) &&
         (D == 128 || D == 256) && R >= 1 &&
         R <= 8 && (R == 1 || R % 2 == 0);
}

cudaError_t launch_verify_int8(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_verify_nvfp4(const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_verify_fp8(const AttnParams &p, int grid, cudaStream_t s);

cudaError_t launch_verify_umma_nvfp4(const AttnParams &p, int max_items, cudaStream_t s);
cudaError_t launch_verify_umma_fp8(const AttnParams &p, int max_items, cudaStream_t s);

// tcgen05 verify (accumulators in tensor memory): NVFP4 / FP8, D = 256
int umma_supported(int dtype, int D, int Q) {
  return (dtype == PA_KV_NVFP4 || dtype == PA_KV_FP8) && D == 256 && Q > 1;
}

cudaError_t launch_verify_umma(const AttnParams &p, int max_items, cudaStream_t s) {
  switch (p.kv.dtype) {
    case PA_KV_NVFP4: return launch_verify_umma_nvfp4(p, max_items, s);
    case PA_KV_FP8: return launch_verify_umma_fp8(p, max_items, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_verify_dense(const AttnParams &p, int grid, cudaStream_t s) {
  switch (p.kv.dtype) {
    case PA_KV_INT8: return launch_verify_int8(p, grid, s);
    case PA_KV_NVFP4: return launch_verify_nvfp4(p, grid, s);
    case PA_KV_FP8: return launch_verify_fp8(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// dense verify tiles (row groups of 16 of the q_len * G rows): quantised
// formats, D = 256
int dense_supported(int dtype, int D, int Q, int G) {
  (void)G;
  return (dtype == PA_KV_INT8 || dtype == PA_KV_NVFP4 || dtype == PA_KV_FP8) && D == 256 && Q > 1;
}

cudaError_t launch_decode_simt(const AttnParams &p, int grid, cudaStream_t s) {
  switch (p.kv.dtype) {
    case PA_KV_BF16: return launch_decode_simt_bf16(p, grid, s);
    case PA_KV_INT8: return launch_decode_simt_int8(p, grid, s);
    case PA_KV_NVFP4: return launch_decode_simt_nvfp4(p, grid, s);
    case PA_KV_FP8: return launch_decode_simt_fp8(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

int simt_supported(int dtype, int D, int R) {
  (void)dtype;
  return (D == 128 || D == 256) && (R == 1 || R == 2 || R == 4 || R == 6 || R == 8);
}
}  // namespace pa

using namespace pa;

namespace {

constexpr int kVersion = 100;
constexpr int kMinSplitBlocks = 8;       // partitions never shorter than 128 tokens (auto mode)
constexpr int kItemCostDecode = 16;      // fixed cost of a work item in key blocks (planner)
constexpr int kItemCostVerify = 32;
// single-launch decode: at most 8 CTAs per cluster (the portable limit), a
// CTA's 4 warps taking up to 2 blocks each in auto mode, and the whole grid
// resident at once (one CTA per SM)
constexpr int kClusterMax = 8;
constexpr int kClusterBlocksPerCta = 8;
constexpr int kClusterMaxCtas = 148;
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Layout {
  size_t hdr = 0, units = 0, prefix_a = 0, prefix_b = 0, items = 0, part_lse = 0, part_o = 0;
  size_t total = 0;
  int U = 0, R = 0, max_items = 0, max_slots = 0;
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Workspace regions for one plan mode.  `target` is the item target the
// call uses (auto: the maximum, so the bound holds for any choice).
// verify row groups: up to kMaxRowGroup rows (a multiple of 16) per group
int group_rows(int Q, int G) { return std::min(kMaxRowGroup, (Q * G + 15) / 16 * 16); }
int row_groups(int Q, int G) { return (Q * G + group_rows(Q, G) - 1) / group_rows(Q, G); }

// mode: 1 virtual (unit per query token), 2 row groups of up to 48 rows
Layout make_layout(const pa_kv_cache *kv, const pa_problem *p, const pa_options *o, int mode) {
  Layout L;
  const int B = p->batch, Q = p->q_len, Hkv = kv->num_kv_heads;
  const int G = p->num_q_heads / Hkv;
  L.U = mode == 1 ? B * Q : B * row_groups(Q, G);
  L.R = mode == 1 ? G : group_rows(Q, G);
  const int maxblk = ceil_div(std::max(p->max_seq_len, 0), kBlock);
  long long items, slots;
  if (o && o->split_blocks > 0) {
    const long long parts = std::max(1, ceil_div(maxblk, o->split_blocks));
    items = (long long)Hkv * L.U * parts;
    slots = (long long)L.U * parts;
  } else {
    const int target = (o && o->target_items > 0) ? std::min(o->target_items, kMaxTargetItems)
                                                  : kMaxTargetItems;
    // one partition per unit beyond the target, plus one more per unit for
    // sequences whose query rows share the longest row's partition bounds
    items = (long long)target + 2LL * Hkv * L.U;
    slots = (long long)ceil_div(target, Hkv) + 2LL * L.U + 1;
    // never more partitions than blocks
    items = std::min(items, (long long)Hkv * L.U * std::max(1, maxblk));
    slots = std::min(slots, (long long)L.U * std::max(1, maxblk));
  }
  L.max_items = (int)std::min<long long>(items, 1LL << 30);
  L.max_slots = (int)std::min<long long>(slots, 1LL << 30);
  size_t off = 0;
  L.hdr = off;
  off += up(kHdrWords * 4);
  L.units = off;
  off += up((size_t)L.U * sizeof(UnitInfo));
  L.prefix_a = off;
  off += up((size_t)L.U * 4);
  L.prefix_b = off;
  off += up((size_t)L.U * 4);
  L.items = off;
  off += up((size_t)L.max_items * sizeof(WorkItem));
  L.part_lse = off;
  off += up((size_t)L.max_slots * Hkv * L.R * 4);
  L.part_o = off;
  off += up((size_t)L.max_slots * Hkv * L.R * kv->head_dim * 4);
  L.total = off;
  return L;
}

int check_kv(const pa_kv_cache *kv) {
  if (!kv) return PA_ERR_INVALID_ARG;
  if (kv->dtype < PA_KV_BF16 || kv->dtype > PA_KV_FP8) return PA_ERR_INVALID_ARG;
  if (kv->block_size != kBlock) return PA_ERR_UNSUPPORTED;
  if (kv->head_dim != 128 && kv->head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (kv->num_kv_heads < 1 || kv->num_blocks < 1) return PA_ERR_INVALID_ARG;
  if (!kv->k_cache || !kv->v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(kv->k_cache) || !aligned16(kv->v_cache)) return PA_ERR_INVALID_ARG;
  if (kv->dtype == PA_KV_INT8 || kv->dtype == PA_KV_NVFP4) {
    if (!kv->k_scale || !kv->v_scale) return PA_ERR_INVALID_ARG;
    if (!aligned16(kv->k_scale) || !aligned16(kv->v_scale)) return PA_ERR_INVALID_ARG;
  }
  if ((kv->dtype == PA_KV_NVFP4 || kv->dtype == PA_KV_FP8) &&
      (!std::isfinite(kv->k_global_scale) || !std::isfinite(kv->v_global_scale)))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

int check_problem(const pa_kv_cache *kv, const pa_problem *p, int max_qlen) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->q_len < 1 || p->max_seq_len < 0) return PA_ERR_INVALID_ARG;
  if (p->q_len > max_qlen) return PA_ERR_UNSUPPORTED;
  if (p->num_q_heads < 1 || p->num_q_heads % kv->num_kv_heads) return PA_ERR_INVALID_ARG;
  const int G = p->num_q_heads / kv->num_kv_heads;
  if (G > kMaxG) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(p->softmax_scale)) return PA_ERR_INVALID_ARG;
  if (p->batch == 0) return PA_OK;
  if (!p->q || !p->block_tables || !p->seq_lens || !p->out) return PA_ERR_INVALID_ARG;
  if (p->block_table_stride < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->out)) return PA_ERR_INVALID_ARG;
  if (!aligned4(p->block_tables) || !aligned4(p->seq_lens)) return PA_ERR_INVALID_ARG;
  if (p->lse_out && !aligned4(p->lse_out)) return PA_ERR_INVALID_ARG;
  if ((long long)p->batch * p->q_len * p->num_q_heads > (1LL << 30)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

KvView view_of(const pa_kv_cache *kv) {
  KvView v;
  v.dtype = kv->dtype;
  v.num_blocks = kv->num_blocks;
  v.hkv = kv->num_kv_heads;
  v.D = kv->head_dim;
  v.k = kv->k_cache;
  v.v = kv->v_cache;
  v.ks = kv->k_scale;
  v.vs = kv->v_scale;
  const bool global = kv->dtype == PA_KV_NVFP4 || kv->dtype == PA_KV_FP8;
  v.kg = global ? kv->k_global_scale : 1.0f;
  v.vg = global ? kv->v_global_scale : 1.0f;
  return v;
}

int run_attention(const pa_kv_cache *kv, const pa_problem *p, const pa_options *o, void *ws,
                  size_t ws_bytes, cudaStream_t stream, bool verify,
                  const uint32_t *extra_err = nullptr) {
  int st = check_kv(kv);
  if (st) return st;
  st = check_problem(kv, p, verify ? kMaxQLen : 1);
  if (st) return st;
  const int kernel = o ? o->kernel : 0;
  if (kernel < 0 || kernel > 5) return PA_ERR_INVALID_ARG;
  if (o && (o->split_blocks < 0 || o->target_items < 0)) return PA_ERR_INVALID_ARG;
  const int test_flags = o ? o->test_flags : 0;
  if (test_flags & ~PA_TEST_EXPIRE_WAIT) return PA_ERR_INVALID_ARG;
  if (p->batch == 0) return PA_OK;
  const int G = p->num_q_heads / kv->num_kv_heads;
  // Kernel choice.  auto: tensor cores (the CUDA cores cannot issue the
  // 3,072 FMA per token and kv head, plus the quantised formats' dequant, at
  // HBM speed; bf16 skewed batch: 1.81 ms against 2.42 ms).  Verify (q_len > 1) on the tensor cores
  // runs as one dense tile of q_len * G rows when supported; otherwise every
  // kernel runs it as a virtual batch (one unit per query token).
  const int Q = p->q_len;
  bool use_tc, dense = false, umma = false, single = false;
  if (kernel == 5) {
    if (verify || Q != 1 || !tc_supported(kv->dtype, kv->head_dim, G) || extra_err)
      return PA_ERR_UNSUPPORTED;
    use_tc = single = true;
  } else if (kernel == 4) {
    if (!umma_supported(kv->dtype, kv->head_dim, Q) || !tc_supported(kv->dtype, kv->head_dim, G))
      return PA_ERR_UNSUPPORTED;
    use_tc = dense = umma = true;
  } else if (kernel == 2 || kernel == 3) {
    if (!tc_supported(kv->dtype, kv->head_dim, G)) return PA_ERR_UNSUPPORTED;
    use_tc = true;
    dense = kernel == 2 && dense_supported(kv->dtype, kv->head_dim, Q, G);
  } else if (kernel == 1) {
    if (!simt_supported(kv->dtype, kv->head_dim, G)) return PA_ERR_UNSUPPORTED;
    use_tc = false;
  } else {
    use_tc = tc_supported(kv->dtype, kv->head_dim, G);
    if (!use_tc && !simt_supported(kv->dtype, kv->head_dim, G)) return PA_ERR_UNSUPPORTED;
    dense = use_tc && dense_supported(kv->dtype, kv->head_dim, Q, G);
    // NVFP4 / FP8 verify: the tcgen05 kernel (4 x 64K keys, 8 queries: NVFP4
    // 0.192 vs 0.304 ms, FP8 0.295 vs 0.298 ms for the mma.sync tiles)
    umma = dense && umma_supported(kv->dtype, kv->head_dim, Q);
  }
  // single-launch decode for small problems (auto mode): every sequence's
  // blocks fit 8 per CTA of a cluster of at most 8, and all clusters run at
  // once; the planner and the merge kernel (two launches) are then pure
  // latency
  const int maxblk_all = ceil_div(std::max(p->max_seq_len, 1), kBlock);
  int cluster = std::min(kClusterMax, std::max(1, ceil_div(maxblk_all, kClusterBlocksPerCta)));
  if (kernel == 0 && use_tc && !dense && !verify && Q == 1 && !extra_err &&
      !(o && (o->split_blocks > 0 || o->target_items > 0)) &&
      maxblk_all <= kClusterMax * kClusterBlocksPerCta &&
      (long long)p->batch * kv->num_kv_heads * cluster <= kClusterMaxCtas)
    single = true;
  // the expired-wait test mode is built into the tensor-core decode kernel only
  if ((test_flags & PA_TEST_EXPIRE_WAIT) && !(use_tc && !dense && !umma)) return PA_ERR_UNSUPPORTED;
  if (single) {
    // no plan, no partials: only the header (error flags, cleared first)
    if (!ws) return PA_ERR_INVALID_ARG;
    if (!aligned16(ws)) return PA_ERR_INVALID_ARG;
    if (ws_bytes < (size_t)kHdrWords * 4) return PA_ERR_WORKSPACE_TOO_SMALL;
    AttnParams ap;
    std::memset(&ap, 0, sizeof ap);
    ap.kv = view_of(kv);
    ap.q = static_cast<const __nv_bfloat16 *>(p->q);
    ap.B = p->batch;
    ap.Q = 1;
    ap.Hq = p->num_q_heads;
    ap.G = G;
    ap.tables = p->block_tables;
    ap.stride = p->block_table_stride;
    ap.seq_lens = p->seq_lens;
    ap.scale_log2 = p->softmax_scale * 1.4426950408889634f;
    ap.out = p->out;
    ap.out_fp32 = p->out_fp32 ? 1 : 0;
    ap.lse_out = p->lse_out;
    ap.hdr = static_cast<uint32_t *>(ws);
    ap.virt = 1;
    ap.RG = 1;
    ap.R = G;
    ap.test_expire = (test_flags & PA_TEST_EXPIRE_WAIT) ? 1 : 0;
    if (cudaMemsetAsync(ws, 0, 16, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (o && o->event_begin &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_begin), stream) != cudaSuccess)
      return PA_ERR_CUDA;
    if (launch_decode_tc_cluster(ap, cluster, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (o && o->event_end &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_end), stream) != cudaSuccess)
      return PA_ERR_CUDA;
    return PA_OK;
  }
  const int mode = dense ? 2 : 1;   // dense verify runs as row groups of up to 48 rows
  const int RG = dense ? row_groups(Q, G) : 1;
  if (!ws) return PA_ERR_INVALID_ARG;
  if (!aligned16(ws)) return PA_ERR_INVALID_ARG;
  const Layout L = make_layout(kv, p, o, mode);
  if (ws_bytes < L.total) return PA_ERR_WORKSPACE_TOO_SMALL;

  uint8_t *w = static_cast<uint8_t *>(ws);
  PlanParams pp;
  std::memset(&pp, 0, sizeof pp);
  pp.seq_lens = p->seq_lens;
  pp.B = p->batch;
  pp.Q = p->q_len;
  pp.virt = mode;
  pp.RG = RG;
  pp.hkv = kv->num_kv_heads;
  pp.capacity = (int)std::min<long long>((long long)p->block_table_stride * kBlock, 1LL << 30);
  // auto target: about 8 items per SM for the one-CTA-per-item kernels; the
  // persistent tcgen05 verify kernel pays a fixed cost per item (its q tile,
  // epilogue and first-tile rescale), so it gets about 2 per SM
  int auto_target = kDefaultTargetItems;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  if (umma && sms > 0) auto_target = std::min(2 * sms, kMaxTargetItems);
  pp.target_items = (o && o->target_items > 0) ? std::min(o->target_items, kMaxTargetItems)
                                               : auto_target;
  // resident CTAs of the attention kernel (the planner rounds equal-length
  // batches to whole rounds of them): one persistent CTA per SM for the
  // tcgen05 verify, the occupancy of the one-CTA-per-item decode kernel.
  // The fixed cost of an item, in key blocks streamed, from sweeps of the
  // item count on equal-length batches: decode (q load, first copies,
  // partial write, merge share) about 16, the tcgen05 verify (its q tile,
  // epilogue and first-tile rescale between items) about 32.
  if (sms > 0 && umma) {
    pp.resident = sms;
    pp.item_cost = kItemCostVerify;
  } else if (sms > 0 && use_tc && !dense) {
    pp.resident = sms * decode_tc_occupancy(kv->dtype, kv->head_dim, L.R);
    pp.item_cost = kItemCostDecode;
  }
  pp.split_blocks = o ? o->split_blocks : 0;
  pp.min_split_blocks = kMinSplitBlocks;
  pp.max_items = L.max_items;
  pp.max_slots = L.max_slots;
  pp.hdr = reinterpret_cast<uint32_t *>(w + L.hdr);
  pp.items = reinterpret_cast<WorkItem *>(w + L.items);
  pp.units = reinterpret_cast<UnitInfo *>(w + L.units);
  pp.prefix_a = reinterpret_cast<int *>(w + L.prefix_a);
  pp.prefix_b = reinterpret_cast<int *>(w + L.prefix_b);
  pp.extra_err = extra_err;

  AttnParams ap;
  std::memset(&ap, 0, sizeof ap);
  ap.kv = view_of(kv);
  ap.q = static_cast<const __nv_bfloat16 *>(p->q);
  ap.B = p->batch;
  ap.Q = p->q_len;
  ap.Hq = p->num_q_heads;
  ap.G = G;
  ap.tables = p->block_tables;
  ap.stride = p->block_table_stride;
  ap.seq_lens = p->seq_lens;
  ap.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  ap.out = p->out;
  ap.out_fp32 = p->out_fp32 ? 1 : 0;
  ap.lse_out = p->lse_out;
  ap.hdr = pp.hdr;
  ap.items = pp.items;
  ap.units = pp.units;
  ap.part_o = reinterpret_cast<float *>(w + L.part_o);
  ap.part_lse = reinterpret_cast<float *>(w + L.part_lse);
  ap.max_items = L.max_items;
  ap.max_slots = L.max_slots;
  ap.virt = mode;
  ap.RG = RG;
  ap.R = L.R;
  ap.test_expire = (test_flags & PA_TEST_EXPIRE_WAIT) ? 1 : 0;

  if (launch_plan(pp, stream) != cudaSuccess) return PA_ERR_CUDA;
  if (o && o->event_begin &&
      cudaEventRecord(static_cast<cudaEvent_t>(o->event_begin), stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if ((umma    ? launch_verify_umma(ap, L.max_items, stream)
       : dense ? launch_verify_dense(ap, L.max_items, stream)
             : use_tc ? launch_decode_tc(ap, L.max_items, stream)
                      : launch_decode_simt(ap, L.max_items, stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  if (o && o->event_end &&
      cudaEventRecord(static_cast<cudaEvent_t>(o->event_end), stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_merge_plan(ap, stream) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

// ---- block-sparse decode: the selection writes a block table per (sequence,
// kv head) into the pool viewed with one kv head per tile; the attention is
// the ordinary decode over that view.
constexpr int kMaxSparseBlocks = 4096;

int check_sparse(const pa_kv_cache *kv, const pa_problem *p, const pa_sparse *sp) {
  if (!sp) return PA_ERR_INVALID_ARG;
  if (sp->sparse_block < kBlock || sp->sparse_block > 256 || sp->sparse_block % kBlock)
    return PA_ERR_UNSUPPORTED;
  if (sp->top_k < 1 || sp->max_sparse_blocks < 1) return PA_ERR_INVALID_ARG;
  if (sp->max_sparse_blocks > kMaxSparseBlocks) return PA_ERR_UNSUPPORTED;
  if ((long long)p->max_seq_len > (long long)sp->max_sparse_blocks * sp->sparse_block)
    return PA_ERR_INVALID_ARG;
  if ((long long)kv->num_blocks * kv->num_kv_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (p->batch > 0 && (!sp->means || !aligned16(sp->means))) return PA_ERR_INVALID_ARG;
  if (sp->selected && !aligned4(sp->selected)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

struct SparseLayout {
  pa_kv_cache kv;        // the view: num_blocks * Hkv tiles of one kv head
  pa_problem prob;       // batch * Hkv virtual sequences of G query heads
  int k_eff, vstride;
  size_t decode_ws, scores, vtables, vlens, err, total;
};

SparseLayout sparse_layout(const pa_kv_cache *kv, const pa_problem *p, const pa_sparse *sp,
                           const pa_options *o) {
  SparseLayout S;
  const int H = kv->num_kv_heads, B = p->batch;
  S.kv = *kv;
  S.kv.num_blocks = kv->num_blocks * H;
  S.kv.num_kv_heads = 1;
  S.k_eff = std::min(sp->top_k, sp->max_sparse_blocks);
  S.vstride = S.k_eff * (sp->sparse_block / kBlock);
  S.prob = *p;
  S.prob.batch = B * H;
  S.prob.num_q_heads = p->num_q_heads / H;
  S.prob.block_table_stride = S.vstride;
  S.prob.max_seq_len = S.k_eff * sp->sparse_block;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  S.decode_ws = up(pa_workspace_bytes(&S.kv, &S.prob, o));
  S.scores = S.decode_ws;
  S.vtables = S.scores + up((size_t)B * H * sp->max_sparse_blocks * 4);
  S.vlens = S.vtables + up((size_t)B * H * S.vstride * 4);
  S.err = S.vlens + up((size_t)B * H * 4);
  S.total = S.err + 256;
  return S;
}

// ---- attention + output projection: o (fp32) in the workspace or the
// caller's fp32 out, then the tensor-core W_O product.
struct WoLayout {
  pa_problem prob;   // with out pointing at o
  int M, K, splits;
  size_t attn_ws, o, part, total;
};

int check_wo(const pa_kv_cache *kv, const pa_problem *p, const pa_wo *wo) {
  if (!wo || !p) return PA_ERR_INVALID_ARG;
  if (wo->hidden < 8 || wo->hidden % 8 || wo->k_split < 0) return PA_ERR_INVALID_ARG;
  if (p->out && !p->out_fp32) return PA_ERR_INVALID_ARG;
  if (p->batch > 0 && (!wo->w || !wo->y || !aligned16(wo->w) || !aligned16(wo->y)))
    return PA_ERR_INVALID_ARG;
  if ((long long)p->num_q_heads * kv->head_dim > (1LL << 24)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

WoLayout wo_layout(const pa_kv_cache *kv, const pa_problem *p, const pa_wo *wo,
                   const pa_options *o) {
  WoLayout W;
  W.prob = *p;
  W.prob.out_fp32 = 1;
  W.M = p->batch * p->q_len;
  W.K = p->num_q_heads * kv->head_dim;
  W.splits = wo_splits(std::max(W.M, 1), W.K, wo->hidden, wo->k_split);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  pa_problem sizing = W.prob;
  const Layout a = make_layout(kv, &sizing, o, 1);
  size_t attn = a.total;
  if (p->q_len > 1) attn = std::max(attn, make_layout(kv, &sizing, o, 2).total);
  W.attn_ws = up(attn);
  W.o = W.attn_ws;
  W.part = W.o + up((size_t)W.M * W.K * 4);
  W.total = W.part + up(W.splits > 1 ? (size_t)W.splits * W.M * wo->hidden * 4 : 0);
  return W;
}

}  // namespace

extern "C" {

size_t pa_decode_wo_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob,
                                    const pa_wo *wo, const pa_options *opt) {
  if (check_kv(kv) != PA_OK || !prob) return 0;
  if (prob->batch < 0 || prob->q_len < 1 || prob->q_len > kMaxQLen || prob->max_seq_len < 0)
    return 0;
  if (prob->num_q_heads < 1 || prob->num_q_heads % kv->num_kv_heads) return 0;
  if (check_wo(kv, prob, wo) != PA_OK) return 0;
  return wo_layout(kv, prob, wo, opt).total;
}

int pa_decode_wo(const pa_kv_cache *kv, const pa_problem *prob, const pa_wo *wo,
                 const pa_options *opt, void *ws, size_t ws_bytes, pa_stream_t stream) {
  int st = check_kv(kv);
  if (st) return st;
  if (!prob) return PA_ERR_INVALID_ARG;
  st = check_wo(kv, prob, wo);
  if (st) return st;
  if (prob->batch == 0) return PA_OK;
  if (!ws || !aligned16(ws)) return PA_ERR_INVALID_ARG;
  WoLayout W = wo_layout(kv, prob, wo, opt);
  if (ws_bytes < W.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t *w = static_cast<uint8_t *>(ws);
  float *o = prob->out ? static_cast<float *>(prob->out) : reinterpret_cast<float *>(w + W.o);
  W.prob.out = o;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = run_attention(kv, &W.prob, opt, ws, W.attn_ws, s, prob->q_len > 1);
  if (st) return st;
  if (launch_wo(o, W.M, W.K, wo->w, wo->hidden, W.splits, reinterpret_cast<float *>(w + W.part),
                wo->y, wo->y_fp32 ? 1 : 0, static_cast<uint32_t *>(ws), s) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_block_means(const pa_kv_cache *kv, const int32_t *block_tables, int32_t stride,
                   const int32_t *seq_lens, const int32_t *first, int32_t count, int32_t batch,
                   int32_t sb, int32_t max_nsb, float *means, void *ws, pa_stream_t stream) {
  int st = check_kv(kv);
  if (st) return st;
  if (batch < 0 || max_nsb < 1 || count < 0) return PA_ERR_INVALID_ARG;
  if (count == 0 || count > max_nsb) count = max_nsb;
  if (sb < kBlock || sb > 256 || sb % kBlock) return PA_ERR_UNSUPPORTED;
  if (batch == 0) return PA_OK;
  if (!block_tables || !seq_lens || !means || stride < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(means) || !aligned4(block_tables) || !aligned4(seq_lens) ||
      (first && !aligned4(first)) || (ws && !aligned16(ws)))
    return PA_ERR_INVALID_ARG;
  uint32_t *hdr = static_cast<uint32_t *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (hdr && cudaMemsetAsync(hdr, 0, 4, s) != cudaSuccess) return PA_ERR_CUDA;
  if (launch_means(view_of(kv), block_tables, stride, seq_lens, first, count, batch, sb, max_nsb,
                   means, hdr, s) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

size_t pa_sparse_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob,
                                 const pa_sparse *sp, const pa_options *opt) {
  if (check_kv(kv) != PA_OK || !prob || prob->q_len != 1 || prob->batch < 0) return 0;
  if (prob->num_q_heads < 1 || prob->num_q_heads % kv->num_kv_heads) return 0;
  if (check_sparse(kv, prob, sp) != PA_OK) return 0;
  const SparseLayout S = sparse_layout(kv, prob, sp, opt);
  return S.decode_ws ? S.total : 0;
}

int pa_decode_sparse(const pa_kv_cache *kv, const pa_problem *prob, const pa_sparse *sp,
                     const pa_options *opt, void *ws, size_t ws_bytes, pa_stream_t stream) {
  int st = check_kv(kv);
  if (st) return st;
  st = check_problem(kv, prob, 1);
  if (st) return st;
  st = check_sparse(kv, prob, sp);
  if (st) return st;
  if (prob->batch == 0) return PA_OK;
  if (!ws || !aligned16(ws)) return PA_ERR_INVALID_ARG;
  const SparseLayout S = sparse_layout(kv, prob, sp, opt);
  if (!S.decode_ws) return PA_ERR_INVALID_ARG;
  if (ws_bytes < S.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *vtables = reinterpret_cast<int *>(w + S.vtables);
  int *vlens = reinterpret_cast<int *>(w + S.vlens);
  uint32_t *err = reinterpret_cast<uint32_t *>(w + S.err);
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess) return PA_ERR_CUDA;
  if (launch_sparse_select(view_of(kv), static_cast<const __nv_bfloat16 *>(prob->q),
                           prob->num_q_heads, prob->block_tables, prob->block_table_stride,
                           prob->seq_lens, prob->batch, sp->sparse_block, sp->max_sparse_blocks,
                           sp->top_k, sp->means, reinterpret_cast<float *>(w + S.scores),
                           sp->selected, vtables, S.vstride, vlens, err, s) != cudaSuccess)
    return PA_ERR_CUDA;
  pa_problem vp = S.prob;
  vp.block_tables = vtables;
  vp.seq_lens = vlens;
  return run_attention(&S.kv, &vp, opt, ws, S.decode_ws, s, false, err);
}


size_t pa_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt) {
  if (check_kv(kv) != PA_OK || !prob) return 0;
  if (prob->batch < 0 || prob->q_len < 1 || prob->q_len > kMaxQLen || prob->max_seq_len < 0)
    return 0;
  if (prob->num_q_heads < 1 || prob->num_q_heads % kv->num_kv_heads) return 0;
  if (opt && (opt->split_blocks < 0 || opt->target_items < 0)) return 0;
  const Layout a = make_layout(kv, prob, opt, 1);
  if (prob->q_len == 1) return a.total;   // decode never uses the row-group layout
  const Layout b = make_layout(kv, prob, opt, 2);
  return std::max(a.total, b.total);
}

int pa_decode(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt, void *ws,
              size_t ws_bytes, pa_stream_t stream) {
  return run_attention(kv, prob, opt, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), false);
}

int pa_verify(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt, void *ws,
              size_t ws_bytes, pa_stream_t stream) {
  return run_attention(kv, prob, opt, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

int pa_merge(const float *part_out, const float *part_lse, int32_t S, int32_t R, int32_t D,
             void *out, int32_t out_fp32, float *lse_out, pa_stream_t stream) {
  if (S < 0 || R < 0 || D < 4 || D % 4 || D > 1024) return PA_ERR_INVALID_ARG;
  if (R == 0) return PA_OK;
  if (!out || (S > 0 && (!part_out || !part_lse))) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || (part_out && !aligned16(part_out)) || (part_lse && !aligned4(part_lse)))
    return PA_ERR_INVALID_ARG;
  if (lse_out && !aligned4(lse_out)) return PA_ERR_INVALID_ARG;
  if (launch_merge_dense(part_out, part_lse, S, R, D, out, out_fp32 ? 1 : 0, lse_out,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_dequant_gather(const pa_kv_cache *kv, const int32_t *block_tables, int32_t stride,
                      const int32_t *seq_lens, int32_t batch, int32_t max_seq_len, float *k_out,
                      float *v_out, void *ws, pa_stream_t stream) {
  int st = check_kv(kv);
  if (st) return st;
  if (batch < 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
  if (batch == 0 || max_seq_len == 0) return PA_OK;
  if (!block_tables || !seq_lens || !k_out || !v_out || stride < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_out) || !aligned16(v_out) || !aligned4(block_tables) || !aligned4(seq_lens))
    return PA_ERR_INVALID_ARG;
  if (ws && !aligned16(ws)) return PA_ERR_INVALID_ARG;
  uint32_t *hdr = static_cast<uint32_t *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (hdr && cudaMemsetAsync(hdr, 0, 4, s) != cudaSuccess) return PA_ERR_CUDA;
  if (launch_gather(view_of(kv), block_tables, stride, seq_lens, batch, max_seq_len, k_out, v_out,
                    hdr, s) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_append_kv(const pa_kv_cache *kv, const void *k_new, const void *v_new, int32_t num_tokens,
                 const int64_t *slot_mapping, void *ws, pa_stream_t stream) {
  int st = check_kv(kv);
  if (st) return st;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if ((long long)num_tokens * kv->num_kv_heads > (1LL << 30)) return PA_ERR_UNSUPPORTED;
  if (ws && !aligned16(ws)) return PA_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!k_new || !v_new || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) ||
        reinterpret_cast<uintptr_t>(slot_mapping) % 8 != 0)
      return PA_ERR_INVALID_ARG;
  }
  uint32_t *hdr = static_cast<uint32_t *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (hdr && cudaMemsetAsync(hdr, 0, 4, s) != cudaSuccess) return PA_ERR_CUDA;
  if (num_tokens == 0) return PA_OK;
  if (launch_append(view_of(kv), k_new, v_new, num_tokens, slot_mapping, hdr, s) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_read_error(const void *ws, uint32_t *host_flags, pa_stream_t stream) {
  if (!ws || !host_flags) return PA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_flags, ws, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

const char *pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_UNKNOWN_STATUS";
}

int pa_version(void) { return kVersion; }

}  // extern "C"
