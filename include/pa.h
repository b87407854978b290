/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV decode attention library.
 *
 * The operation (PagedAttention decode; Kwon et al., "Efficient Memory
 * Management for Large Language Model Serving with PagedAttention", cited
 * on "vLLM Fork with focus on GB10 Homelabs", section "About"): each
 * sequence b owns a list of fixed-size physical KV blocks; logical token t
 * lives in block  block_tables[b][t / 16]  at slot  t % 16.  For every
 * query token i < q_len and query head h (kv head h / G, G = Hq / Hkv):
 *
 *     n   = seq_lens[b] - q_len + 1 + i        (keys visible to query i)
 *     s_t = softmax_scale * <q[b,i,h,:], K_t>  for t < n
 *     out[b,i,h,:] = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m),  m = max s
 *     lse[b,i,h]   = m + ln sum_t exp(s_t - m)          (natural log)
 *
 * q_len = 1 is decode.  q_len > 1 is speculative verify: the q_len new
 * tokens are the last q_len keys already written to the cache and each
 * sees the prior context plus the new tokens up to itself (the "virtual
 * batch for speculative positions" of "vLLM-SM70", section "Why"; 8 query
 * tokens = DFlash2 K=7 on "vLLM All-NVFP4 DFlash2 for Blackwell", section
 * "What makes this stack different").  Keys are split into partitions that
 * run in parallel and are combined with a log-sum-exp merge ("split-KV
 * merge", "vLLM Fork with focus on GB10 Homelabs", "Acknowledgments").
 *
 * KV storage formats (dequantised in registers inside the kernels):
 *   PA_KV_BF16  : k/v bf16 [NB, Hkv, 16, D]; no scales.
 *   PA_KV_INT8  : k/v int8 [NB, Hkv, 16, D]; k/v_scale fp16 [NB, Hkv, 16]
 *                 (one scale per token and kv head); value = code * scale
 *                 ("vLLM-SM70", "Why": int8 KV cache).
 *   PA_KV_NVFP4 : k/v uint8 [NB, Hkv, 16, D/2], E2M1 codes, element 2i in
 *                 the low nibble; k/v_scale uint8 [NB, Hkv, 16, D/16], one
 *                 FP8-E4M3 scale per 16 consecutive head-dim elements;
 *                 k/v_global_scale fp32 per tensor; value =
 *                 (e2m1(code) * e4m3(scale)) * global  ("vLLM All-NVFP4
 *                 DFlash2 for Blackwell", "What makes this stack
 *                 different": NVFP4 KV cache; UE4M3 block scales: "vLLM
 *                 Fork with focus on GB10 Homelabs", "Acknowledgments").
 *   PA_KV_FP8   : k/v uint8 [NB, Hkv, 16, D], FP8-E4M3 codes; no scale tensors;
 *                 k/v_global_scale fp32 per tensor; value = e4m3(code) * global
 *                 (FP8 KV with inline dequant: "vLLM Fork with focus on GB10
 *                 Homelabs", "Acknowledgments"; "vLLM All-NVFP4 DFlash2 for
 *                 Blackwell", "What makes this stack different").
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless marked (host).  Every data
 *     pointer must be 16-byte aligned.  The caller owns every buffer; the
 *     library never allocates, never synchronises (except pa_read_error)
 *     and keeps no state between calls: it is reentrant and thread-safe,
 *     and a call can be captured in a CUDA graph (no host reads of device
 *     data; the split plan is computed on the device).
 *   - All work is enqueued asynchronously on `stream` (NULL = legacy
 *     default stream).
 *   - Argument errors are detected on the host and return a negative
 *     pa_status with NOTHING launched.  A failed launch returns
 *     PA_ERR_CUDA.
 *   - Errors that only the device can see (a block-table entry outside
 *     [0, num_blocks), seq_len < 0 or beyond the table's capacity, a
 *     verify row with seq_len < q_len) never trap: the offending block is
 *     skipped or the length clamped, and a bit is set in the workspace
 *     header, which pa_read_error returns.  The flags describe the most
 *     recent pa_decode / pa_verify call that used the workspace.
 *   - seq_lens[b] = 0 marks a padded row: its outputs are 0 and lse -inf.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *pa_stream_t;   /* same type as cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1,          /* null pointer, bad size, misalignment */
  PA_ERR_UNSUPPORTED = -2,          /* head_dim, block_size, G or q_len not built */
  PA_ERR_WORKSPACE_TOO_SMALL = -3,  /* ws_bytes < pa_workspace_bytes(...) */
  PA_ERR_CUDA = -4                  /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_INT8 = 1, PA_KV_NVFP4 = 2, PA_KV_FP8 = 3 } pa_kv_dtype;

/* Device error flags (pa_read_error). */
#define PA_ERRF_BAD_BLOCK_ID      0x1u  /* table entry outside [0, num_blocks): block skipped */
#define PA_ERRF_LEN_OVER_CAPACITY 0x2u  /* seq_len > 16 * block_table_stride: clamped */
#define PA_ERRF_NEG_LEN           0x4u  /* seq_len < 0: treated as 0 */
#define PA_ERRF_LEN_LT_QLEN       0x8u  /* verify: 0 < seq_len < q_len: rows with no key get 0 */
#define PA_ERRF_WAIT_TIMEOUT      0x10u /* an in-kernel wait hit its iteration cap: outputs invalid */
#define PA_ERRF_PLAN_OVERFLOW     0x20u /* the split plan did not fit the workspace: nothing computed */
#define PA_ERRF_BAD_SLOT          0x40u /* pa_append_kv: slot outside [-1, 16 * num_blocks): row skipped */

/* The paged KV pool.  block_size must be 16; head_dim 128 or 256. */
typedef struct pa_kv_cache {
  int32_t dtype;          /* pa_kv_dtype */
  int32_t num_blocks;     /* NB, physical blocks in the pool */
  int32_t block_size;     /* tokens per block (16) */
  int32_t num_kv_heads;   /* Hkv */
  int32_t head_dim;       /* D */
  const void *k_cache;    /* layouts: see the format list above */
  const void *v_cache;
  const void *k_scale;    /* NULL for bf16 and FP8 */
  const void *v_scale;
  float k_global_scale;   /* (host) NVFP4 / FP8 per-tensor scale; ignored otherwise */
  float v_global_scale;
} pa_kv_cache;

/* One batched call. */
typedef struct pa_problem {
  int32_t batch;               /* B >= 0 */
  int32_t num_q_heads;         /* Hq, a multiple of num_kv_heads; Hq / Hkv <= 8 */
  int32_t q_len;               /* 1 for pa_decode; 1..16 for pa_verify */
  const void *q;               /* bf16 [B, q_len, Hq, D] */
  const int32_t *block_tables; /* int32 [B, block_table_stride] physical block ids */
  int32_t block_table_stride;  /* >= 1 entries per row; capacity = 16 * stride tokens */
  const int32_t *seq_lens;     /* int32 [B] keys in the cache per sequence, including
                                  the q_len new ones; 0 = padded row */
  int32_t max_seq_len;         /* (host) upper bound of seq_lens, sizes the workspace */
  float softmax_scale;         /* multiplies q.k, e.g. 1/sqrt(D) */
  void *out;                   /* bf16 (or fp32 if out_fp32) [B, q_len, Hq, D] */
  int32_t out_fp32;            /* 0: bf16 round-to-nearest-even output; 1: fp32 */
  float *lse_out;              /* optional fp32 [B, q_len, Hq] natural-log LSE, or NULL */
} pa_problem;

/* Optional knobs; pass NULL for defaults. */
typedef struct pa_options {
  int32_t kernel;          /* 0 auto: decode (every format) -> 2, or 5 for a small problem;
                              int8 verify (head_dim 256) -> 2 (dense tiles);
                              bf16 verify -> 2 (one unit per query token);
                              NVFP4 / FP8 verify (head_dim 256) -> 4.
                              1 CUDA-core (SIMT) kernel; 2 tensor-core kernel (mma.sync;
                              bf16 fragments by ldmatrix; verify: dense tiles of up to
                              48 of the q_len * G rows when the format is
                              int8/NVFP4/FP8 and head_dim 256); 3
                              tensor-core kernel with verify run as one unit per query
                              token; 4 verify on the tcgen05 tensor cores (accumulators
                              in tensor memory; NVFP4 / FP8, head_dim 256, q_len > 1;
                              else PA_ERR_UNSUPPORTED); 5 single-launch decode (pa_decode
                              only): one cluster of up to 8 CTAs per (sequence, kv head),
                              no planner and no merge kernel, the partials merged in
                              distributed shared memory; auto mode picks it when every
                              sequence has at most 1,024 keys (max_seq_len) and batch x
                              kv heads x cluster size <= 148.  It uses only the first
                              256 bytes of the workspace. */
  int32_t split_blocks;    /* 0 auto; >0 = fixed number of 16-token blocks per partition
                              (a value >= the longest sequence's block count disables
                              split-K) */
  int32_t target_items;    /* 0 auto; >0 = aim for about this many work items */
  void *event_begin;       /* optional cudaEvent_t recorded just before the attention
                              kernel (after the planner) -- for timing that kernel */
  void *event_end;         /* optional cudaEvent_t recorded just after it */
  int32_t test_flags;      /* 0 normally.  PA_TEST_EXPIRE_WAIT (tensor-core decode,
                              kernel 2 or auto decode; else PA_ERR_UNSUPPORTED): every warp
                              of the attention kernel withholds the copy of its first KV
                              block, so its wait for that block runs out after a short cap
                              (about a thousand polls); the kernel then records
                              PA_ERRF_WAIT_TIMEOUT, lets the copies it did issue land and
                              returns.  The outputs of such a call are meaningless.  It
                              exercises the capped-wait failure path without faulting or
                              hanging the GPU.  Other bits: PA_ERR_INVALID_ARG. */
} pa_options;

#define PA_TEST_EXPIRE_WAIT 0x1

/* Bytes of device workspace a pa_decode / pa_verify call with these
 * arguments needs (an upper bound computed from batch, q_len, heads and
 * max_seq_len only).  The workspace needs no initialisation; it may be
 * reused by consecutive calls on the same stream, never by two calls that
 * can run at the same time.  Returns 0 on invalid arguments. */
size_t pa_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt);

/* Decode (q_len == 1): out = attention of q over the paged cache.
 * ws: device workspace of ws_bytes >= pa_workspace_bytes(...). */
int pa_decode(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt,
              void *ws, size_t ws_bytes, pa_stream_t stream);

/* Decode without a caller-provided workspace, for callers that cannot
 * allocate device memory (code whose framework owns every device
 * allocation, plugins handed only their input and output buffers, hosts
 * that forbid cudaMalloc after start-up).  The split-K workspace lives in a
 * fixed device array of PA_NOALLOC_SCRATCH_BYTES inside the library, held
 * by every GPU that loads it until the process exits; nothing is allocated
 * per call.  The PagedAttention paper has no counterpart to this entry
 * point.  Same arguments, semantics, status codes and results as pa_decode
 * with default options.  Returns PA_ERR_WORKSPACE_TOO_SMALL, with nothing
 * launched, when the call would need more workspace than
 * PA_NOALLOC_SCRATCH_BYTES (about (2 * batch + 300) * Hkv * G * D * 4 bytes
 * for the default plan).  The first call on each device (with that device
 * current) looks up the array's device address and keeps it; make that
 * first call before any stream capture.  The kept address is that of the
 * device's current primary context: after cudaDeviceReset, do not call this
 * entry point on that device again in the same process.  All calls share
 * the array: calls that can overlap on the GPU race.  The device error
 * flags of these calls cannot be read back. */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_decode_noalloc(const pa_kv_cache *kv, const pa_problem *prob, pa_stream_t stream);

/* Speculative verify (1 <= q_len <= 16), causal among the q_len new tokens
 * (query i sees keys t < seq_len - q_len + 1 + i).  Requires seq_len >=
 * q_len or 0; other rows set PA_ERRF_LEN_LT_QLEN. */
int pa_verify(const pa_kv_cache *kv, const pa_problem *prob, const pa_options *opt,
              void *ws, size_t ws_bytes, pa_stream_t stream);

/* Log-sum-exp merge of S partial attention results over disjoint key sets
 * (split-KV merge, "vLLM Fork with focus on GB10 Homelabs",
 * "Acknowledgments"):
 *   part_out fp32 [S, R, D] (each partial normalised by its own weights),
 *   part_lse fp32 [S, R] natural-log LSE, -inf marks an empty partial.
 *   out[r,:] = sum_p exp(lse_p - M) part_out[p,r,:] / sum_p exp(lse_p - M),
 *   M = max_p lse_p;  lse_out[r] = M + ln sum_p exp(lse_p - M) (optional).
 * A row whose partials are all empty gets 0 and -inf.  out is bf16 or
 * fp32 (out_fp32) [R, D].  D <= 1024, a multiple of 4. */
int pa_merge(const float *part_out, const float *part_lse, int32_t S, int32_t R, int32_t D,
             void *out, int32_t out_fp32, float *lse_out, pa_stream_t stream);

/* Debug: gathers through the block table and dequantises exactly as the
 * attention kernels do, writing fp32 k_out / v_out [B, Hkv, max_seq_len, D]
 * (positions t >= seq_len, and blocks with an out-of-range id, are 0).
 * The values are bit-exact: bf16 widened; int8 (float)code * (float)scale;
 * NVFP4 fp32_round((e2m1 * e4m3) * global); FP8 fp32_round(e4m3 * global).  ws may be NULL; if given (>=
 * 256 bytes) its header receives the device error flags. */
int pa_dequant_gather(const pa_kv_cache *kv, const int32_t *block_tables,
                      int32_t block_table_stride, const int32_t *seq_lens, int32_t batch,
                      int32_t max_seq_len, float *k_out, float *v_out, void *ws,
                      pa_stream_t stream);

/* Block-sparse decode by per-block mean keys ("vLLM-SM70", "Known
 * limitations" and its production fixes: sparse-decode selection over
 * per-block mean keys, 64-token blocks, at most 4096 of them, mean keys
 * refreshed for every request of a decode batch).  Sparse block j of a
 * sequence holds logical tokens [j * sparse_block, (j + 1) * sparse_block).
 * Its mean key is the mean of the dequantised keys of its valid tokens; for
 * kv head h it scores max over the query heads of h of q . mean_j; the
 * top_k blocks of largest score (ties to the lower index) are attended
 * exactly, each kv head over its own selection. */
typedef struct pa_sparse {
  int32_t sparse_block;       /* tokens per sparse block: a multiple of 16, 16..256 */
  int32_t top_k;              /* sparse blocks attended per (sequence, kv head), >= 1 */
  int32_t max_sparse_blocks;  /* second axis of means, 1..4096, and at least
                                 ceil(max_seq_len / sparse_block) */
  const float *means;         /* fp32 [batch, max_sparse_blocks, num_kv_heads, head_dim] */
  int32_t *selected;          /* optional out: int32 [batch, num_kv_heads, top_k], the
                                 selected sparse blocks in ascending order, -1 padded */
} pa_sparse;

/* Mean keys of sparse blocks first_sparse_block[b] .. first_sparse_block[b]
 * + count - 1 of every sequence (those that hold keys) into means (layout
 * as in pa_sparse; other entries are not written).  first_sparse_block
 * (int32 [batch]) may be NULL (= 0); count = 0 means max_sparse_blocks.  A
 * decode step refreshes each sequence's last sparse block (count 1),
 * prefill all of them.  ws: NULL, or >= 256 bytes whose header receives the
 * flags. */
int pa_block_means(const pa_kv_cache *kv, const int32_t *block_tables,
                   int32_t block_table_stride, const int32_t *seq_lens,
                   const int32_t *first_sparse_block, int32_t count, int32_t batch,
                   int32_t sparse_block, int32_t max_sparse_blocks, float *means, void *ws,
                   pa_stream_t stream);

/* Workspace of pa_decode_sparse (0 on invalid arguments). */
size_t pa_sparse_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob,
                                 const pa_sparse *sp, const pa_options *opt);

/* Block-sparse decode (q_len 1): scores and selects the sparse blocks on the
 * device, then runs pa_decode over the selected blocks of each kv head
 * (the pool viewed as [num_blocks * num_kv_heads, 1, 16, head_dim], one
 * virtual sequence per (sequence, kv head)).  Outputs as pa_decode; the
 * workspace header (pa_read_error) also collects the selection's flags
 * (PA_ERRF_PLAN_OVERFLOW: a sequence longer than max_sparse_blocks sparse
 * blocks, attended over its first max_sparse_blocks only). */
int pa_decode_sparse(const pa_kv_cache *kv, const pa_problem *prob, const pa_sparse *sp,
                     const pa_options *opt, void *ws, size_t ws_bytes, pa_stream_t stream);

/* Attention followed by the output projection in the same call: for every
 * query token, y[token, :] = o[token, :] . W_O with o that token's output
 * of all num_q_heads heads flattened (index head * head_dim + d) ("vLLM
 * Fork with focus on GB10 Homelabs", "Roadmap": fused attention + W_O
 * GEMV, K-parallel split).  W_O is bf16 [num_q_heads * head_dim, hidden]
 * row-major; y is [batch * q_len, hidden], bf16 or fp32 (y_fp32).  hidden
 * must be a multiple of 8.  prob->out may be NULL (o then stays in the
 * workspace); if given it must be fp32 (out_fp32 = 1) and receives o.
 * q_len > 1 runs the verify attention.  k_split: 0 = automatic. */
typedef struct pa_wo {
  const void *w;        /* bf16 [num_q_heads * head_dim, hidden], 16-byte aligned */
  int32_t hidden;
  void *y;
  int32_t y_fp32;
  int32_t k_split;
} pa_wo;

size_t pa_decode_wo_workspace_bytes(const pa_kv_cache *kv, const pa_problem *prob,
                                    const pa_wo *wo, const pa_options *opt);
int pa_decode_wo(const pa_kv_cache *kv, const pa_problem *prob, const pa_wo *wo,
                 const pa_options *opt, void *ws, size_t ws_bytes, pa_stream_t stream);

/* KV append: quantise-on-write of the new tokens' K and V into the pool --
 * the write side of the paged cache (PagedAttention, "vLLM Fork with focus
 * on GB10 Homelabs", "About"): row (t, h) goes to block slot_mapping[t] / 16,
 * offset slot_mapping[t] % 16, kv head h.  A padded row carries slot -1 and
 * writes nothing ("vLLM-SM70", "Known limitations": padded drafter rows
 * once wrote K/V into other requests' slots).
 *   kv            the pool; its code and scale arrays are WRITTEN (the const
 *                 of pa_kv_cache's pointers is cast away).  NVFP4 / FP8 use
 *                 k_global_scale / v_global_scale as the pool's fixed
 *                 per-tensor scales (a scale <= 0 writes zero codes).
 *   k_new, v_new  bf16 [num_tokens, num_kv_heads, head_dim], 16-byte aligned.
 *   slot_mapping  int64 [num_tokens], 8-byte aligned: block * 16 + offset,
 *                 or -1.  Slots must be distinct within one call (two rows
 *                 for one slot leave that slot's bytes unspecified).  A slot
 *                 outside [-1, 16 * num_blocks) is skipped and sets
 *                 PA_ERRF_BAD_SLOT.
 *   ws            NULL, or >= 256 bytes whose header receives the flags.
 * Encoding (every rounding decision in fp32, round to nearest even):
 *   bf16  : copied.
 *   int8  : s = fp16(amax / 127) over the (token, kv head) row; code =
 *           clamp(rint(x / s), -127, 127); s = 0 gives 0.
 *   FP8   : code = E4M3 nearest to |x / g| (saturating at 448) with the
 *           sign of x / g, except that a zero magnitude is written +0.
 *   NVFP4 : per 16 elements, scale = E4M3 nearest to amax16 / (g * 6);
 *           code = E2M1 nearest to |x / (e4m3(scale) * g)| (saturating at 6)
 *           with the sign bit of that quotient; element 2i in the low
 *           nibble.
 * num_tokens = 0 launches nothing but the flag reset.  Returns PA_OK,
 * PA_ERR_INVALID_ARG (null pointer, misalignment, num_tokens < 0),
 * PA_ERR_UNSUPPORTED (head_dim, block_size) or PA_ERR_CUDA. */
int pa_append_kv(const pa_kv_cache *kv, const void *k_new, const void *v_new, int32_t num_tokens,
                 const int64_t *slot_mapping, void *ws, pa_stream_t stream);

/* Copies the device error flags (PA_ERRF_*) of the last call that used ws
 * to *host_flags (host).  Synchronises `stream`. */
int pa_read_error(const void *ws, uint32_t *host_flags, pa_stream_t stream);

/* Human-readable name of a pa_status value (static string). */
const char *pa_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
