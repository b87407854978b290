/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged-KV decode and
 * speculative-verify attention, and for the split-K log-sum-exp merge.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the plain definition of the method):
 *   PagedAttention (Kwon et al., "Efficient Memory Management for Large
 *   Language Model Serving with PagedAttention", cited on "vLLM Fork with
 *   focus on GB10 Homelabs", section "About"): the keys and values of a
 *   sequence live in fixed-size physical blocks; logical token t of
 *   sequence b sits in block  block_tables[b][t / block_size]  at slot
 *   t % block_size.  Decode attention is exact softmax attention of the new
 *   query over those keys; "vLLM-SM70", section "Why", checks every kernel
 *   against such an exact-softmax oracle (fp32 there, fp64 here).
 *
 *   For sequence b, query token i < Q and query head h (kv head h / G):
 *     n   = L_b - Q + 1 + i         (speculative verify: query i sees the
 *                                    prior context and new tokens 0..i --
 *                                    the "virtual batch" reading of
 *                                    "vLLM-SM70", "Why"; decode: n = L_b)
 *     s_t = scale * sum_d q[d] * k_t[d]          for t < n
 *     m   = max_t s_t,  w_t = exp(s_t - m)
 *     o   = sum_t w_t v_t / sum_t w_t,  lse = m + log(sum_t w_t)
 *   L_b = 0 (a padded row) gives o = 0 and lse = -inf.
 *
 *   Split-K ("split-KV merge", "vLLM Fork with focus on GB10 Homelabs",
 *   "Acknowledgments"): partial results (o_p, lse_p) over disjoint key
 *   ranges combine as  M = max lse_p,  w_p = exp(lse_p - M),
 *   o = sum w_p o_p / sum w_p,  lse = M + log sum w_p.
 *
 * Storage formats, decoded here from their bit-field definitions:
 *   bf16  : the fp32 whose upper 16 bits are the code.
 *   int8  : value = (float)code * (float)scale, scale an IEEE fp16 per
 *           (token, kv head)  ("vLLM-SM70": int8 KV cache).
 *   NVFP4 : value = RN_fp32( (e2m1(code) * e4m3(scale)) * g ), one E4M3
 *           scale per 16 consecutive head-dim elements and one fp32 g per
 *           cache tensor ("vLLM All-NVFP4 DFlash2 for Blackwell", "What
 *           makes this stack different": NVFP4 KV cache; UE4M3 block
 *           scales: "vLLM Fork with focus on GB10 Homelabs",
 *           "Acknowledgments").  Element 2i of a byte pair is the low
 *           nibble.  e2m1 * e4m3 is exact in fp32, so the value is one
 *           fp32 rounding of the product with g -- block scale first.
 *   FP8   : value = RN_fp32( e4m3(code) * g ), one fp32 g per cache tensor
 *           (FP8 KV with inline dequant, "vLLM Fork with focus on GB10
 *           Homelabs", "Acknowledgments").
 *   The fp32 dequantised value is widened to double for the attention.
 *
 *   Block-sparse decode ("vLLM-SM70", "Known limitations" and the
 *   production fixes: sparse-decode selection over per-block mean keys,
 *   blocks of 64 tokens, at most 4096 of them): the mean key of sparse
 *   block j is the mean of the dequantised keys of its valid tokens; block
 *   j of kv head h scores max over the query heads of h of q . mean_j;
 *   the top_k blocks (ties to the lower index) are attended exactly
 *   (oracle_block_means, oracle_sparse_select, oracle_attend_sparse).
 *
 *   KV append (quantise-on-write): new K / V rows of a step go to the
 *   slots that a slot mapping names, slot = block * block_size + offset;
 *   a padded row carries slot -1 and writes nothing ("vLLM-SM70", "Known
 *   limitations": padded drafter rows once wrote K/V into other requests'
 *   slots).  The encoders invert the decoders above, rounding to the
 *   nearest point of each format's grid with ties to the even code
 *   (oracle_append below).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -pthread
 *        (no fast-math: the fp32 dequant must round exactly once).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_BF16 = 0, OR_INT8 = 1, OR_NVFP4 = 2, OR_FP8 = 3 };

typedef struct {
  int32_t dtype;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  const void *k_cache, *v_cache;
  const void *k_scale, *v_scale;
  float k_global, v_global;
} oracle_cache;

/* ---------------------------------------------------------------- formats */

double oracle_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_fp16_value(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);                 /* (m / 2^10) * 2^-14 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/2^10) * 2^(e-15) */
  return s ? -v : v;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN; max 448, min subnormal 2^-9. */
double oracle_e4m3_value(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xf, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);                  /* (m/8) * 2^-6 */
  else
    v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* OCP FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit. */
double oracle_e2m1_value(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* fp32 value of element d of token slot (blk, head, slot); which = 0 K, 1 V */
static float dequant(const oracle_cache *c, int which, int64_t blk, int head, int slot, int d) {
  const int64_t row = (blk * c->num_kv_heads + head) * c->block_size + slot;
  const int D = c->head_dim;
  const void *data = which ? c->v_cache : c->k_cache;
  const void *scale = which ? c->v_scale : c->k_scale;
  switch (c->dtype) {
    case OR_BF16:
      return (float)oracle_bf16_value(((const uint16_t *)data)[row * D + d]);
    case OR_INT8: {
      float code = (float)((const int8_t *)data)[row * D + d];
      float s = (float)oracle_fp16_value(((const uint16_t *)scale)[row]);
      return code * s;
    }
    case OR_NVFP4: {
      uint8_t byte = ((const uint8_t *)data)[row * (D / 2) + d / 2];
      uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
      uint8_t sc = ((const uint8_t *)scale)[row * (D / 16) + d / 16];
      float prod = (float)(oracle_e2m1_value(code) * oracle_e4m3_value(sc));
      float g = which ? c->v_global : c->k_global;
      return prod * g;
    }
    case OR_FP8: {
      float e = (float)oracle_e4m3_value(((const uint8_t *)data)[row * D + d]);
      float g = which ? c->v_global : c->k_global;
      return e * g;
    }
  }
  return NAN;
}

/* Dequantised row (D floats) of logical token t of sequence b; returns 0 and
 * writes zeros if the table entry is out of range. */
static int token_row(const oracle_cache *c, int which, const int32_t *tables, int32_t stride,
                     int b, int t, int head, float *out) {
  int32_t blk = tables[(int64_t)b * stride + t / c->block_size];
  if (blk < 0 || blk >= c->num_blocks) {
    for (int d = 0; d < c->head_dim; ++d) out[d] = 0.0f;
    return 0;
  }
  for (int d = 0; d < c->head_dim; ++d)
    out[d] = dequant(c, which, blk, head, t % c->block_size, d);
  return 1;
}

/* Dequantised K and V through the block table, [B, Hkv, max_len, D] fp32;
 * positions t >= seq_len are zero. */
void oracle_gather(const oracle_cache *c, const int32_t *tables, int32_t stride,
                   const int32_t *seq_lens, int32_t B, int32_t max_len, float *k_out, float *v_out) {
  const int D = c->head_dim, H = c->num_kv_heads;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int t = 0; t < max_len; ++t) {
        int64_t off = (((int64_t)b * H + h) * max_len + t) * D;
        if (t < seq_lens[b]) {
          token_row(c, 0, tables, stride, b, t, h, k_out + off);
          token_row(c, 1, tables, stride, b, t, h, v_out + off);
        } else {
          for (int d = 0; d < D; ++d) k_out[off + d] = v_out[off + d] = 0.0f;
        }
      }
}

/* ------------------------------------------------------------ attention */

typedef struct {
  const oracle_cache *c;
  const uint16_t *q;          /* bf16 bits [B, Q, Hq, D] */
  int32_t B, Q, Hq;
  const int32_t *tables;
  int32_t stride;
  const int32_t *seq_lens;
  const int32_t *key_begin;   /* optional [B]: first key index considered */
  const int32_t *key_end;     /* optional [B]: one past the last key considered */
  double scale;
  double *out;                /* [B, Q, Hq, D] */
  double *lse;                /* [B, Q, Hq] */
  const int32_t *items;       /* optional list of (b, kv_head) pairs */
  int32_t nitems;
  int32_t next;               /* shared work counter */
  pthread_mutex_t mu;
} attend_job;

static void attend_item(attend_job *J, int b, int kvh, double *scores, float *row, double *acc) {
  const oracle_cache *c = J->c;
  const int D = c->head_dim, Q = J->Q, Hq = J->Hq;
  const int G = Hq / c->num_kv_heads;
  const int R = Q * G;
  const int L = J->seq_lens[b];
  int lo = J->key_begin ? J->key_begin[b] : 0;
  int hi_all = J->key_end ? J->key_end[b] : L;
  if (lo < 0) lo = 0;
  if (hi_all > L) hi_all = L;

  /* query vectors, exact bf16 -> double */
  double *qv = (double *)malloc(sizeof(double) * (size_t)R * D);
  int *n = (int *)malloc(sizeof(int) * R);
  for (int i = 0; i < Q; ++i)
    for (int g = 0; g < G; ++g) {
      int h = kvh * G + g, r = i * G + g;
      const uint16_t *qs = J->q + (((int64_t)b * Q + i) * Hq + h) * D;
      for (int d = 0; d < D; ++d) qv[(int64_t)r * D + d] = oracle_bf16_value(qs[d]);
      int lim = L - Q + 1 + i; /* keys visible to query token i */
      if (L == 0) lim = 0;
      if (lim > hi_all) lim = hi_all;
      n[r] = lim;
    }
  int tmax = 0;
  for (int r = 0; r < R; ++r) if (n[r] > tmax) tmax = n[r];

  /* pass 1: scores */
  for (int t = lo; t < tmax; ++t) {
    token_row(c, 0, J->tables, J->stride, b, t, kvh, row);
    for (int r = 0; r < R; ++r) {
      if (t >= n[r]) continue;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qv[(int64_t)r * D + d] * (double)row[d];
      scores[(int64_t)r * tmax + t] = J->scale * dot;
    }
  }
  /* pass 2: max */
  double *mx = (double *)malloc(sizeof(double) * R);
  double *sum = (double *)malloc(sizeof(double) * R);
  for (int r = 0; r < R; ++r) {
    mx[r] = -INFINITY;
    sum[r] = 0.0;
    for (int t = lo; t < n[r]; ++t)
      if (scores[(int64_t)r * tmax + t] > mx[r]) mx[r] = scores[(int64_t)r * tmax + t];
  }
  /* pass 3: weights and values */
  memset(acc, 0, sizeof(double) * (size_t)R * D);
  for (int t = lo; t < tmax; ++t) {
    token_row(c, 1, J->tables, J->stride, b, t, kvh, row);
    for (int r = 0; r < R; ++r) {
      if (t >= n[r]) continue;
      double w = exp(scores[(int64_t)r * tmax + t] - mx[r]);
      sum[r] += w;
      for (int d = 0; d < D; ++d) acc[(int64_t)r * D + d] += w * (double)row[d];
    }
  }
  for (int i = 0; i < Q; ++i)
    for (int g = 0; g < G; ++g) {
      int h = kvh * G + g, r = i * G + g;
      int64_t o = (((int64_t)b * Q + i) * Hq + h);
      if (n[r] <= lo || sum[r] == 0.0) {
        for (int d = 0; d < D; ++d) J->out[o * D + d] = 0.0;
        J->lse[o] = -INFINITY;
      } else {
        for (int d = 0; d < D; ++d) J->out[o * D + d] = acc[(int64_t)r * D + d] / sum[r];
        J->lse[o] = mx[r] + log(sum[r]);
      }
    }
  free(qv);
  free(n);
  free(mx);
  free(sum);
}

static void *attend_worker(void *arg) {
  attend_job *J = (attend_job *)arg;
  const oracle_cache *c = J->c;
  const int D = c->head_dim, G = J->Hq / c->num_kv_heads, R = J->Q * G;
  int lmax = 1;
  for (int b = 0; b < J->B; ++b) if (J->seq_lens[b] > lmax) lmax = J->seq_lens[b];
  double *scores = (double *)malloc(sizeof(double) * (size_t)R * lmax);
  float *row = (float *)malloc(sizeof(float) * D);
  double *acc = (double *)malloc(sizeof(double) * (size_t)R * D);
  const int total = J->items ? J->nitems : J->B * c->num_kv_heads;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int it = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (it >= total) break;
    int b, kvh;
    if (J->items) {
      b = J->items[2 * it];
      kvh = J->items[2 * it + 1];
    } else {
      b = it / c->num_kv_heads;
      kvh = it % c->num_kv_heads;
    }
    attend_item(J, b, kvh, scores, row, acc);
  }
  free(scores);
  free(row);
  free(acc);
  return NULL;
}

/* Exact attention for every (b, query token, query head), or only for the
 * (b, kv head) pairs listed in `items` (nitems pairs) when items != NULL.
 * key_begin / key_end (optional, [B]) restrict the keys to a sub-range,
 * which yields the partial (o, lse) of one split.  Returns 0. */
int oracle_attend(const oracle_cache *c, const uint16_t *q, int32_t B, int32_t Q, int32_t Hq,
                  const int32_t *tables, int32_t stride, const int32_t *seq_lens,
                  const int32_t *key_begin, const int32_t *key_end, double scale,
                  double *out, double *lse, const int32_t *items, int32_t nitems,
                  int32_t nthreads) {
  attend_job J;
  memset(&J, 0, sizeof J);
  J.c = c; J.q = q; J.B = B; J.Q = Q; J.Hq = Hq; J.tables = tables; J.stride = stride;
  J.seq_lens = seq_lens; J.key_begin = key_begin; J.key_end = key_end; J.scale = scale;
  J.out = out; J.lse = lse; J.items = items; J.nitems = nitems; J.next = 0;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, attend_worker, &J);
  attend_worker(&J);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/* Log-sum-exp merge of S partials: part_o [S, R, D], part_lse [S, R]
 * (-inf marks an empty partial) -> out [R, D], lse [R]. */
void oracle_merge(const double *part_o, const double *part_lse, int32_t S, int32_t R, int32_t D,
                  double *out, double *lse) {
  for (int r = 0; r < R; ++r) {
    double M = -INFINITY;
    for (int p = 0; p < S; ++p)
      if (part_lse[(int64_t)p * R + r] > M) M = part_lse[(int64_t)p * R + r];
    if (M == -INFINITY) {
      for (int d = 0; d < D; ++d) out[(int64_t)r * D + d] = 0.0;
      lse[r] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int d = 0; d < D; ++d) out[(int64_t)r * D + d] = 0.0;
    for (int p = 0; p < S; ++p) {
      double l = part_lse[(int64_t)p * R + r];
      if (l == -INFINITY) continue;
      double w = exp(l - M);
      wsum += w;
      for (int d = 0; d < D; ++d)
        out[(int64_t)r * D + d] += w * part_o[((int64_t)p * R + r) * D + d];
    }
    for (int d = 0; d < D; ++d) out[(int64_t)r * D + d] /= wsum;
    lse[r] = M + log(wsum);
  }
}

/* ------------------------------------------------------------ KV append */

/* Nearest of the grid values val(0) < val(1) < ... < val(n-1) to a >= 0,
 * ties to the even code; a beyond the last value gives the last code
 * (saturation).  Binary search for the last code not above a, then the
 * nearer of it and its successor. */
static int round_to_grid(double a, double (*val)(int), int n) {
  if (a >= val(n - 1)) return n - 1;
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (val(mid) <= a) lo = mid; else hi = mid - 1;
  }
  double below = a - val(lo), above = val(lo + 1) - a;
  if (below < above) return lo;
  if (above < below) return lo + 1;
  return (lo & 1) ? lo + 1 : lo;
}

/* non-negative grids: E4M3 codes 0..126 (127 is NaN), E2M1 codes 0..7, and
 * binary16 codes 0..0x7C00 with the infinity code standing at 2^16, where
 * IEEE round-to-nearest-even sends everything from 65520 up */
static double e4m3_grid(int c) { return oracle_e4m3_value((uint8_t)c); }
static double e2m1_grid(int c) { return oracle_e2m1_value((uint8_t)c); }
static double fp16_grid(int c) { return c == 0x7C00 ? 65536.0 : oracle_fp16_value((uint16_t)c); }

/* round half to even of a double holding an fp32 quotient */
static double round_half_even(double q) {
  double f = floor(q), frac = q - f;
  if (frac > 0.5) return f + 1.0;
  if (frac < 0.5) return f;
  return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* Encode one (token, kv head) row of D bf16 values into cache row `row` of
 * tensor `which` (0 K, 1 V).  Formats (readings of the pages' formats):
 *   bf16  : the bits are copied.
 *   int8  : s = fp16_RNE(amax / 127) with amax / 127 in fp32; code =
 *           clamp(RNE(x / s), -127, 127) with x / s in fp32; s = 0 gives 0.
 *   FP8   : y = x / g in fp32; code = nearest E4M3 to |y| (saturating at
 *           448), sign bit when y < 0 and the magnitude code is not 0;
 *           g <= 0 gives 0.
 *   NVFP4 : per 16 elements t = amax16 / (g * 6) in fp32 (g * 6 rounded
 *           first); scale = nearest E4M3 to t; sg = e4m3(scale) * g in
 *           fp32; y = x / sg in fp32 (0 when sg = 0); code = nearest E2M1
 *           to |y| (saturating at 6) with the sign of y in bit 3; element
 *           2i in the low nibble. */
static void encode_row(const oracle_cache *c, int which, int64_t row, const uint16_t *src) {
  const int D = c->head_dim;
  void *data = (void *)(which ? c->v_cache : c->k_cache);
  void *scale = (void *)(which ? c->v_scale : c->k_scale);
  const float g = which ? c->v_global : c->k_global;
  float *x = (float *)malloc(sizeof(float) * D);
  for (int d = 0; d < D; ++d) x[d] = (float)oracle_bf16_value(src[d]);
  switch (c->dtype) {
    case OR_BF16:
      for (int d = 0; d < D; ++d) ((uint16_t *)data)[row * D + d] = src[d];
      break;
    case OR_INT8: {
      float amax = 0.0f;
      for (int d = 0; d < D; ++d) if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
      float ratio = amax / 127.0f;
      uint16_t s16 = (uint16_t)round_to_grid((double)ratio, fp16_grid, 0x7C01);
      ((uint16_t *)scale)[row] = s16;
      float s = (float)oracle_fp16_value(s16);
      for (int d = 0; d < D; ++d) {
        double code = 0.0;
        if (s > 0.0f) {
          float q = x[d] / s;
          code = round_half_even((double)q);
          if (code > 127.0) code = 127.0;
          if (code < -127.0) code = -127.0;
        }
        ((int8_t *)data)[row * D + d] = (int8_t)code;
      }
      break;
    }
    case OR_FP8:
      for (int d = 0; d < D; ++d) {
        float y = g > 0.0f ? x[d] / g : 0.0f;
        int mag = round_to_grid(fabs((double)y), e4m3_grid, 127);
        ((uint8_t *)data)[row * D + d] = (uint8_t)(mag | ((y < 0.0f && mag != 0) ? 0x80 : 0));
      }
      break;
    case OR_NVFP4:
      for (int j = 0; j < D / 16; ++j) {
        float amax = 0.0f;
        for (int e = 0; e < 16; ++e) if (fabsf(x[16 * j + e]) > amax) amax = fabsf(x[16 * j + e]);
        float denom = g * 6.0f;
        float t = g > 0.0f ? amax / denom : 0.0f;
        int sc = round_to_grid((double)t, e4m3_grid, 127);
        ((uint8_t *)scale)[row * (D / 16) + j] = (uint8_t)sc;
        float sval = (float)oracle_e4m3_value((uint8_t)sc);
        float sg = sval * g;
        for (int e = 0; e < 16; e += 2) {
          uint8_t nib[2];
          for (int k = 0; k < 2; ++k) {
            float y = sg > 0.0f ? x[16 * j + e + k] / sg : 0.0f;
            int mag = round_to_grid(fabs((double)y), e2m1_grid, 8);
            nib[k] = (uint8_t)(mag | (signbit(y) ? 8 : 0));
          }
          ((uint8_t *)data)[row * (D / 2) + (16 * j + e) / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
        }
      }
      break;
  }
  free(x);
}

/* Append T new tokens: k_new / v_new bf16 bits [T, Hkv, D]; slot_mapping[t]
 * = physical block * block_size + offset, or -1 for a padded row (nothing
 * written).  A slot outside [-1, num_blocks * block_size) is skipped and
 * counted; returns that count.  Slots are assumed distinct. */
int oracle_append(const oracle_cache *c, const uint16_t *k_new, const uint16_t *v_new, int32_t T,
                  const int64_t *slot_mapping) {
  const int H = c->num_kv_heads, D = c->head_dim, bs = c->block_size;
  const int64_t nslots = (int64_t)c->num_blocks * bs;
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < -1 || slot >= nslots) {
      ++bad;
      continue;
    }
    int64_t blk = slot / bs, off = slot % bs;
    for (int h = 0; h < H; ++h) {
      int64_t row = (blk * H + h) * bs + off;
      encode_row(c, 0, row, k_new + ((int64_t)t * H + h) * D);
      encode_row(c, 1, row, v_new + ((int64_t)t * H + h) * D);
    }
  }
  return bad;
}

/* ------------------------------------------------- block-sparse decode */

/* means [B, max_nsb, Hkv, D]: sparse block j of sequence b covers logical
 * tokens [j * sb, min((j + 1) * sb, L)); its mean key is the mean of their
 * dequantised keys.  Blocks past the sequence are 0. */
void oracle_block_means(const oracle_cache *c, const int32_t *tables, int32_t stride,
                        const int32_t *seq_lens, int32_t B, int32_t sb, int32_t max_nsb,
                        double *means) {
  const int H = c->num_kv_heads, D = c->head_dim;
  float *row = (float *)malloc(sizeof(float) * D);
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < max_nsb; ++j)
      for (int h = 0; h < H; ++h) {
        double *m = means + (((int64_t)b * max_nsb + j) * H + h) * D;
        for (int d = 0; d < D; ++d) m[d] = 0.0;
        int lo = j * sb, hi = (j + 1) * sb;
        if (hi > seq_lens[b]) hi = seq_lens[b];
        if (lo >= hi) continue;
        for (int t = lo; t < hi; ++t) {
          token_row(c, 0, tables, stride, b, t, h, row);
          for (int d = 0; d < D; ++d) m[d] += (double)row[d];
        }
        for (int d = 0; d < D; ++d) m[d] /= (double)(hi - lo);
      }
  free(row);
}

/* scores [B, Hkv, max_nsb]: score of block j for kv head h = max over the
 * query heads of h of q . mean_j (q bf16 [B, 1, Hq, D]); blocks j >= nsb[b]
 * score -inf.  sel [B, Hkv, k]: the min(k, nsb[b]) blocks of largest score,
 * ties to the lower index, in ascending block order, then -1. */
void oracle_sparse_select(const uint16_t *q, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                          const double *means, const int32_t *nsb, int32_t max_nsb, int32_t k,
                          double *scores, int32_t *sel) {
  const int G = Hq / Hkv;
  char *taken = (char *)malloc(max_nsb > 0 ? max_nsb : 1);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      double *sc = scores + ((int64_t)b * Hkv + h) * max_nsb;
      for (int j = 0; j < max_nsb; ++j) {
        sc[j] = -INFINITY;
        if (j >= nsb[b]) continue;
        const double *m = means + (((int64_t)b * max_nsb + j) * Hkv + h) * D;
        for (int g = 0; g < G; ++g) {
          const uint16_t *qh = q + ((int64_t)b * Hq + h * G + g) * D;
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += oracle_bf16_value(qh[d]) * m[d];
          if (dot > sc[j]) sc[j] = dot;
        }
      }
      /* k rounds of "largest remaining score, lowest index on ties" */
      int n = nsb[b] < k ? nsb[b] : k;
      memset(taken, 0, max_nsb > 0 ? max_nsb : 1);
      for (int r = 0; r < n; ++r) {
        int best = -1;
        for (int j = 0; j < nsb[b]; ++j)
          if (!taken[j] && (best < 0 || sc[j] > sc[best])) best = j;
        taken[best] = 1;
      }
      int32_t *out = sel + ((int64_t)b * Hkv + h) * k;
      int pos = 0;
      for (int j = 0; j < nsb[b]; ++j)
        if (taken[j]) out[pos++] = j;
      for (; pos < k; ++pos) out[pos] = -1;
    }
  free(taken);
}

/* Exact decode attention (Q = 1) of every query head over the keys of the
 * sparse blocks its kv head selected (sel as above, sparse block size sb).
 * out [B, 1, Hq, D], lse [B, 1, Hq]; a head with no key gets 0 and -inf. */
void oracle_attend_sparse(const oracle_cache *c, const uint16_t *q, int32_t B, int32_t Hq,
                          const int32_t *tables, int32_t stride, const int32_t *seq_lens,
                          const int32_t *sel, int32_t k, int32_t sb, double scale, double *out,
                          double *lse) {
  const int H = c->num_kv_heads, D = c->head_dim, G = Hq / H;
  float *row = (float *)malloc(sizeof(float) * D);
  int lmax = 1;
  for (int b = 0; b < B; ++b) if (seq_lens[b] > lmax) lmax = seq_lens[b];
  double *s = (double *)malloc(sizeof(double) * lmax);
  char *keep = (char *)malloc(lmax);
  double *acc = (double *)malloc(sizeof(double) * D);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      const int L = seq_lens[b];
      memset(keep, 0, lmax);
      for (int r = 0; r < k; ++r) {
        int j = sel[((int64_t)b * H + h) * k + r];
        if (j < 0) continue;
        for (int t = j * sb; t < (j + 1) * sb && t < L; ++t) keep[t] = 1;
      }
      for (int g = 0; g < G; ++g) {
        const int qh = h * G + g;
        const uint16_t *qv = q + ((int64_t)b * Hq + qh) * D;
        double m = -INFINITY;
        for (int t = 0; t < L; ++t) {
          if (!keep[t]) continue;
          token_row(c, 0, tables, stride, b, t, h, row);
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += oracle_bf16_value(qv[d]) * (double)row[d];
          s[t] = scale * dot;
          if (s[t] > m) m = s[t];
        }
        double sum = 0.0;
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int t = 0; t < L; ++t) {
          if (!keep[t]) continue;
          double w = exp(s[t] - m);
          sum += w;
          token_row(c, 1, tables, stride, b, t, h, row);
          for (int d = 0; d < D; ++d) acc[d] += w * (double)row[d];
        }
        double *o = out + ((int64_t)b * Hq + qh) * D;
        if (sum == 0.0) {
          for (int d = 0; d < D; ++d) o[d] = 0.0;
          lse[(int64_t)b * Hq + qh] = -INFINITY;
        } else {
          for (int d = 0; d < D; ++d) o[d] = acc[d] / sum;
          lse[(int64_t)b * Hq + qh] = m + log(sum);
        }
      }
    }
  free(row);
  free(s);
  free(keep);
  free(acc);
}
