/*
 * paged_ref.c -- plain fp64 CPU oracle for batched paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no source, header, helper or table with the CUDA
 * library; the two meet only in the bytes the seeded input generator draws.
 *
 * What it computes follows the PhotonInfer README (page
 * "openaitx.github.io/.../photon_infer/README-ko.html"):
 *   - "Key features / GPU-optimized kernels": batched paged attention over a
 *     block-wise KV cache, softmax computed in a numerically stable way;
 *   - "Technical details / Paged attention": block-wise KV cache, per-sequence
 *     cache offsets, one batched cache-write operation for many sequences;
 *   - "Key features / GPU-optimized kernels": batched RoPE among the fused
 *     operations (ref_rope: rotate-half form, theta_k = pos * base^(-2k/d),
 *     the plain reading of the rotary embedding; the page names no variant).
 * The page prints no formula.  Its plain reading, used here, is scaled
 * dot-product attention of one query row per sequence over that sequence's
 * cached keys/values, with grouped query heads:
 *     s_j   = scale * sum_i q[b][h][i] * K_j[kvh][i],      kvh = h / (Hq/Hkv)
 *     out   = sum_j exp(s_j - max_j s_j) V_j / sum_j exp(s_j - max_j s_j)
 * with j running over the logical positions 0 .. context_len-1, each found
 * through the block table (physical block = table[j / bs], row = j % bs).
 *
 * Everything is evaluated in double: inputs are widened exactly (fp16 and
 * bf16 are decoded from their IEEE bit fields), sums run in logical order
 * j = 0, 1, ... with no blocking and no splitting.  The split-partition merge
 * (ref_merge) is provided separately so tests can check that the direct sum
 * equals the log-sum-exp combination of sub-range results.
 *
 * Storage dtypes: 0 = fp32, 1 = fp16, 2 = bf16 (raw 16-bit patterns).
 * Layouts (row-major):
 *   q, out        [B][Hq][d]
 *   k_cache, v    [NB][Hkv][bs][d]
 *   block_tables  int32 [B][MBS], padding -1 (never read past ceil(ctx/bs))
 *   slot_mapping  int64 [T], slot = block * bs + offset, negative = skip
 *   k_new, v_new  [T][Hkv][d]
 *   dense gather  [B][Hkv][MBS*bs][d], zero past the context
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { REF_OK = 0, REF_BAD_ARG = -1, REF_BAD_SLOT = -2, REF_DUP_SLOT = -3,
       REF_BAD_BLOCK = -4, REF_BAD_CTX = -5 };

static size_t elem_size(int dtype) { return dtype == 0 ? 4u : 2u; }

/* IEEE binary16 -> double, from the bit fields (exact). */
static double f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1f;
  int man = h & 0x3ff;
  double v;
  if (ex == 0)
    v = ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
  else if (ex == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexp((double)(man | 0x400), ex - 25);   /* 1.man * 2^(ex-15)      */
  return sign ? -v : v;
}

/* bfloat16 -> double: the high half of an IEEE binary32 (exact). */
static double bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

static double load(const void* base, size_t idx, int dtype) {
  if (dtype == 0) {
    float f;
    memcpy(&f, (const char*)base + idx * 4, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + idx * 2, 2);
  return dtype == 1 ? f16_to_double(h) : bf16_to_double(h);
}

/* ---------------------------------------------------------------- cache write
 * For every new row t and KV head h with slot_t >= 0, copy the d raw elements
 * of k_new[t][h] and v_new[t][h] to cache[slot_t / bs][h][slot_t % bs]. A bit
 * copy: no conversion.  Slots outside [0, NB*bs) and duplicated slots are
 * rejected before anything is written. */
int ref_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                    int32_t num_tokens, void* k_cache, void* v_cache, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, int32_t num_blocks, int32_t dtype) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return REF_BAD_ARG;
  const int64_t nslots = (int64_t)num_blocks * block_size;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s >= nslots) return REF_BAD_SLOT;
    if (s < 0) continue;
    for (int32_t u = 0; u < t; ++u)
      if (slot_mapping[u] == s) return REF_DUP_SLOT;
  }
  const size_t e = elem_size(dtype);
  const size_t row = (size_t)head_dim * e;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    int64_t blk = s / block_size, off = s % block_size;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      size_t src = ((size_t)t * num_kv_heads + h) * row;
      size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row;
      memcpy((char*)k_cache + dst, (const char*)k_new + src, row);
      memcpy((char*)v_cache + dst, (const char*)v_new + src, row);
    }
  }
  return REF_OK;
}

/* ---------------------------------------------------------------- gather
 * dense[b][h][j] = cache[block_tables[b][j / bs]][h][j % bs] for j < ctx_b,
 * zero bytes for ctx_b <= j < MBS*bs.  A bit copy. */
int ref_gather(const void* k_cache, const void* v_cache, const int32_t* block_tables,
               const int32_t* context_lens, void* k_dense, void* v_dense, int32_t num_seqs,
               int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
               int32_t max_blocks_per_seq, int32_t dtype) {
  const size_t e = elem_size(dtype);
  const size_t row = (size_t)head_dim * e;
  const int64_t span = (int64_t)max_blocks_per_seq * block_size;
  for (int32_t b = 0; b < num_seqs; ++b) {
    int32_t ctx = context_lens[b];
    if (ctx < 0 || ctx > span) return REF_BAD_CTX;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int64_t j = 0; j < span; ++j) {
        size_t dst = (((size_t)b * num_kv_heads + h) * span + j) * row;
        if (j >= ctx) {
          memset((char*)k_dense + dst, 0, row);
          memset((char*)v_dense + dst, 0, row);
          continue;
        }
        int32_t blk = block_tables[(size_t)b * max_blocks_per_seq + j / block_size];
        if (blk < 0 || blk >= num_blocks) return REF_BAD_BLOCK;
        size_t src = (((size_t)blk * num_kv_heads + h) * block_size + j % block_size) * row;
        memcpy((char*)k_dense + dst, (const char*)k_cache + src, row);
        memcpy((char*)v_dense + dst, (const char*)v_cache + src, row);
      }
    }
  }
  return REF_OK;
}

/* ---------------------------------------------------------------- attention */
typedef struct {
  const void *q, *k_cache, *v_cache;
  const double* q64;  /* optional: query rows already in double (then q is unused) */
  const int32_t *block_tables, *context_lens;
  double scale;
  int32_t B, Hq, Hkv, d, bs, NB, MBS, dtype;
} ref_problem;

/* Offset of element 0 of logical row j of sequence b, KV head kvh, or -1 when
 * the table entry is outside the pool. */
static int64_t row_offset(const ref_problem* P, int32_t b, int32_t kvh, int64_t j) {
  int32_t blk = P->block_tables[(size_t)b * P->MBS + j / P->bs];
  if (blk < 0 || blk >= P->NB) return -1;
  return ((((int64_t)blk * P->Hkv + kvh) * P->bs) + j % P->bs) * P->d;
}

/* Unnormalised partial over logical positions [j0, j1) for (b, h):
 *   m = max s_j,  l = sum exp(s_j - m),  o = sum exp(s_j - m) V_j.
 * An empty range gives m = -inf, l = 0, o = 0.  Two passes, plain order. */
static int attend_range(const ref_problem* P, int32_t b, int32_t h, int64_t j0, int64_t j1,
                        double* m_out, double* l_out, double* o, double* s /* scratch */) {
  const int32_t G = P->Hq / P->Hkv;
  const int32_t kvh = h / G;
  const int32_t d = P->d;
  const size_t qoff = ((size_t)b * P->Hq + h) * d;
  for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
  double m = -INFINITY;
  for (int64_t j = j0; j < j1; ++j) {
    int64_t r = row_offset(P, b, kvh, j);
    if (r < 0) return REF_BAD_BLOCK;
    double dot = 0.0;
    for (int32_t i = 0; i < d; ++i) {
      const double qi = P->q64 ? P->q64[qoff + i] : load(P->q, qoff + i, P->dtype);
      dot += qi * load(P->k_cache, (size_t)r + i, P->dtype);
    }
    s[j - j0] = P->scale * dot;
    if (s[j - j0] > m) m = s[j - j0];
  }
  double l = 0.0;
  for (int64_t j = j0; j < j1; ++j) {
    double p = exp(s[j - j0] - m);
    l += p;
    int64_t r = row_offset(P, b, kvh, j);
    for (int32_t i = 0; i < d; ++i) o[i] += p * load(P->v_cache, (size_t)r + i, P->dtype);
  }
  *m_out = m;
  *l_out = l;
  return REF_OK;
}

/* out[b][h][:] = softmax over the whole context, written as doubles.  A
 * context of length 0 gives an all-zero row. */
static int attend_one(const ref_problem* P, int32_t b, int32_t h, double* out, double* s) {
  int32_t ctx = P->context_lens[b];
  double m, l;
  int rc = attend_range(P, b, h, 0, ctx, &m, &l, out, s);
  if (rc) return rc;
  if (ctx == 0) return REF_OK;
  for (int32_t i = 0; i < P->d; ++i) out[i] /= l;
  return REF_OK;
}

typedef struct {
  const ref_problem* P;
  double* out;
  int32_t first, stride;  /* work items (b, kvh) handled by this thread */
  int rc;
} worker_arg;

static void* worker(void* argp) {
  worker_arg* a = (worker_arg*)argp;
  const ref_problem* P = a->P;
  const int32_t G = P->Hq / P->Hkv;
  double* s = (double*)malloc(sizeof(double) * ((size_t)P->MBS * P->bs + 1));
  if (!s) { a->rc = REF_BAD_ARG; return NULL; }
  a->rc = REF_OK;
  for (int32_t w = a->first; w < P->B * P->Hkv; w += a->stride) {
    int32_t b = w / P->Hkv, kvh = w % P->Hkv;
    for (int32_t g = 0; g < G; ++g) {
      int32_t h = kvh * G + g;
      int rc = attend_one(P, b, h, a->out + ((size_t)b * P->Hq + h) * P->d, s);
      if (rc) a->rc = rc;
    }
  }
  free(s);
  return NULL;
}

static int check_problem(const ref_problem* P) {
  if (P->B < 0 || P->Hq <= 0 || P->Hkv <= 0 || P->Hq % P->Hkv || P->d <= 0 || P->bs <= 0 ||
      P->MBS <= 0 || P->dtype < 0 || P->dtype > 2)
    return REF_BAD_ARG;
  for (int32_t b = 0; b < P->B; ++b)
    if (P->context_lens[b] < 0 || P->context_lens[b] > (int64_t)P->MBS * P->bs) return REF_BAD_CTX;
  return REF_OK;
}

/* Full decode: out[B][Hq][d] as double.  num_threads > 1 spreads the (b, kvh)
 * work items over POSIX threads; the arithmetic per item is unchanged. */
int ref_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens, double scale,
                     double* out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     int32_t max_blocks_per_seq, int32_t dtype, int32_t num_threads) {
  ref_problem P = {q, k_cache, v_cache, NULL, block_tables, context_lens, scale, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, dtype};
  int rc = check_problem(&P);
  if (rc) return rc;
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  pthread_t tid[256];
  worker_arg args[256];
  for (int32_t t = 0; t < num_threads; ++t) {
    args[t].P = &P;
    args[t].out = out;
    args[t].first = t;
    args[t].stride = num_threads;
    args[t].rc = REF_OK;
  }
  if (num_threads == 1) {
    worker(&args[0]);
    return args[0].rc;
  }
  int32_t started = 0;
  for (int32_t t = 0; t < num_threads; ++t) {
    if (pthread_create(&tid[t], NULL, worker, &args[t]) != 0) break;
    ++started;
  }
  /* Any thread that failed to start: do its share here. */
  for (int32_t t = started; t < num_threads; ++t) worker(&args[t]);
  for (int32_t t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  for (int32_t t = 0; t < num_threads; ++t)
    if (args[t].rc) return args[t].rc;
  return REF_OK;
}

/* One (b, h) output row; for sampled checks on large problems. */
int ref_paged_decode_row(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens, double scale,
                         int32_t b, int32_t h, double* out_row, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_blocks, int32_t max_blocks_per_seq,
                         int32_t dtype) {
  ref_problem P = {q, k_cache, v_cache, NULL, block_tables, context_lens, scale, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, dtype};
  int rc = check_problem(&P);
  if (rc) return rc;
  if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) return REF_BAD_ARG;
  double* s = (double*)malloc(sizeof(double) * ((size_t)max_blocks_per_seq * block_size + 1));
  if (!s) return REF_BAD_ARG;
  rc = attend_one(&P, b, h, out_row, s);
  free(s);
  return rc;
}

/* Partial (m, l, unnormalised o) over logical positions [j0, j1) of (b, h). */
int ref_attend_range(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens, double scale,
                     int32_t b, int32_t h, int64_t j0, int64_t j1, double* m, double* l,
                     double* o, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     int32_t max_blocks_per_seq, int32_t dtype) {
  ref_problem P = {q, k_cache, v_cache, NULL, block_tables, context_lens, scale, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, dtype};
  int rc = check_problem(&P);
  if (rc) return rc;
  if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads || j0 < 0 || j1 < j0 ||
      j1 > context_lens[b])
    return REF_BAD_ARG;
  double* s = (double*)malloc(sizeof(double) * ((size_t)(j1 - j0) + 1));
  if (!s) return REF_BAD_ARG;
  rc = attend_range(&P, b, h, j0, j1, m, l, o, s);
  free(s);
  return rc;
}

/* Log-sum-exp merge of P partials (m_p, l_p, o_p[d]):
 *   M = max over partials with l_p > 0 of m_p
 *   out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p
 * Partials with l_p = 0 (empty ranges) are skipped; if all are empty the
 * result is zero. */
void ref_merge(int32_t num_parts, const double* m, const double* l, const double* o,
               int32_t head_dim, double* out) {
  double M = -INFINITY;
  for (int32_t p = 0; p < num_parts; ++p)
    if (l[p] > 0.0 && m[p] > M) M = m[p];
  for (int32_t i = 0; i < head_dim; ++i) out[i] = 0.0;
  if (M == -INFINITY) return;
  double den = 0.0;
  for (int32_t p = 0; p < num_parts; ++p) {
    if (!(l[p] > 0.0)) continue;
    double w = exp(m[p] - M);
    den += w * l[p];
    for (int32_t i = 0; i < head_dim; ++i) out[i] += w * o[(size_t)p * head_dim + i];
  }
  for (int32_t i = 0; i < head_dim; ++i) out[i] /= den;
}

/* Exact widening of stored elements to double (lets tests read fp16/bf16
 * pools without relying on any other decoder). */
void ref_widen(const void* src, size_t n, int32_t dtype, double* dst) {
  for (size_t i = 0; i < n; ++i) dst[i] = load(src, i, dtype);
}

/* ---------------------------------------------------------------- RoPE
 * Rotary position embedding, rotate-half form (the Llama / Qwen convention;
 * the README's "Key features / GPU-optimized kernels" lists batched RoPE among
 * the fused operations, without a formula).  For k < d/2, with
 * theta_k = pos * base^(-2k/d):
 *   y[k]       = x[k] cos(theta_k) - x[k + d/2] sin(theta_k)
 *   y[k + d/2] = x[k + d/2] cos(theta_k) + x[k] sin(theta_k)
 * In double, on already-widened values. */
void ref_rope(const double* x, int32_t head_dim, int64_t pos, double base, double* y) {
  const int32_t half = head_dim / 2;
  for (int32_t k = 0; k < half; ++k) {
    const double theta = (double)pos * pow(base, -2.0 * (double)k / (double)head_dim);
    const double c = cos(theta), s = sin(theta);
    const double a = x[k], b = x[k + half];
    y[k] = a * c - b * s;
    y[k + half] = b * c + a * s;
  }
}

/* ref_paged_decode with the query rows given in double (used for rotated
 * queries, which are never stored). */
int ref_paged_decode_q64(const double* q64, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens, double scale,
                         double* out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         int32_t max_blocks_per_seq, int32_t dtype, int32_t num_threads) {
  ref_problem P = {NULL, k_cache, v_cache, q64, block_tables, context_lens, scale, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, dtype};
  int rc = check_problem(&P);
  if (rc) return rc;
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  pthread_t tid[256];
  worker_arg args[256];
  for (int32_t t = 0; t < num_threads; ++t) {
    args[t].P = &P;
    args[t].out = out;
    args[t].first = t;
    args[t].stride = num_threads;
    args[t].rc = REF_OK;
  }
  int32_t started = 0;
  for (int32_t t = 1; t < num_threads; ++t) {
    if (pthread_create(&tid[t], NULL, worker, &args[t]) != 0) break;
    ++started;
  }
  worker(&args[0]);
  for (int32_t t = 1 + started; t < num_threads; ++t) worker(&args[t]);
  for (int32_t t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  for (int32_t t = 0; t < num_threads; ++t)
    if (args[t].rc) return args[t].rc;
  return REF_OK;
}
