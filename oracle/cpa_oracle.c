/*
 * cpa_oracle.c -- plain fp64 CPU oracle for one chunked-prefill attention step
 * over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * loads it.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *
 *   For sequence s with q_len = query_start_loc[s+1] - query_start_loc[s]
 *   and ctx = seq_lens[s] (tokens in the cache after this step's append),
 *   query row i (0 <= i < q_len) of head h sees the keys j = 0 .. ctx-q_len+i.
 *     - "vllm-learning-book 05. Chunked Prefill", section 3 (chunked attention
 *       correctness): a chunk's queries see every earlier chunk's K/V already
 *       in the cache plus a causal mask inside the chunk; Q&A of section 8:
 *       the K/V include the tokens the current chunk has just written.
 *     - "Chunked Prefill 技术深度解析", section 4.1: a chunk never sees the
 *       K/V of later chunks.
 *     - "How Chunked Prefill Stops Decode Starvation", "The fix": each chunk
 *       attends to all previous chunks of the same prompt.
 *   A decode is the case q_len = 1, which sees all ctx keys.
 *
 *   logits  x_j = scale * <q_{i,h}, K_j>           (standard scaled dot product)
 *   weights p_j = exp(x_j - max_k x_k) / sum_k exp(x_k - max_k x_k)
 *   output  o   = sum_j p_j V_j
 *
 *   GQA head map (the pages are silent; contiguous groups are adopted):
 *     kv_head = h / (Hq / Hkv).
 *
 * Paged cache layout ("Chunked Prefill 技术深度解析", section 4.2: fixed pages
 * of 16 tokens, each request owning a list of pages): separate K and V caches,
 * each [num_pages][Hkv][page_size][D].  Logical position j of sequence s lives
 * in page block_table[s][j / page_size] at offset j % page_size.
 *
 * Inputs are the exact stored values widened to double: fp32, bf16 or IEEE
 * binary16 queries and caches, or an 8-bit cache of OCP FP8 E4M3 codes whose
 * values are multiplied by a per-tensor scale (k_scale for K, v_scale for V).
 * The pages do not cover an 8-bit cache; the format, its rounding and the
 * scale follow the OCP 8-bit Floating Point Specification (OFP8), E4M3: 1 sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent
 * field 0, no infinities, S.1111.111 the only NaN, largest finite 448.
 * All arithmetic is in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_E4M3 = 3 };

/* IEEE 754 binary16: sign, 5-bit exponent with bias 15, 10-bit fraction;
 * exponent field 0 holds zero and the subnormals (fraction * 2^-24), 31 the
 * infinities and NaNs. */
static double f16_value(uint16_t h) {
  int sign = h >> 15, ef = (h >> 10) & 31, fr = h & 1023;
  double v;
  if (ef == 31) v = fr ? NAN : INFINITY;
  else if (ef == 0) v = ldexp((double)fr, -24);
  else v = ldexp((double)(1024 + fr), ef - 25);
  return sign ? -v : v;
}

/* OFP8 E4M3: exponent field 0 holds zero and the subnormals (mantissa * 2^-9);
 * otherwise (8 + mantissa) * 2^(exponent field - 10); S.1111.111 is NaN. */
static double e4m3_value(uint8_t b) {
  int sign = b >> 7, ef = (b >> 3) & 15, m = b & 7;
  if (ef == 15 && m == 7) return NAN;
  double v = ef == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), ef - 10);
  return sign ? -v : v;
}

/* Elements of the 16-bit IEEE and 8-bit formats (kept out of line so that the
 * bf16 and fp32 loads below stay small enough to inline in the dot loops). */
static double __attribute__((noinline)) load_narrow(const void *base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F16) return f16_value(((const uint16_t *)base)[idx]);
  return e4m3_value(((const uint8_t *)base)[idx]);
}

/* One stored element widened to double (exact for every format here).  bf16
 * is the upper half of an IEEE binary32. */
static double load_elem(const void *base, int dtype, int64_t idx) {
  if (dtype == ORACLE_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
  return load_narrow(base, dtype, idx);
}

/* OFP8 E4M3 code of a binary32 value: round to nearest, ties to even, at the
 * spacing of the value's binade (the subnormal spacing 2^-9 below 2^-6), and
 * saturate to +-448 (magnitudes that round past 448, and infinities); NaN
 * gives the NaN code 0x7f.  With e = max(floor(log2|y|), -6) and
 * m = |y| / 2^(e-3) rounded to an integer, the code is 8 (e + 6) + m: this
 * covers subnormals (e = -6, m < 8) and a mantissa that rounds up into the
 * next binade (m = 16) alike. */
static uint8_t e4m3_code(float y) {
  if (isnan(y)) return 0x7f;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7e;
  int e = -6;
  if (a > 0.0) {
    int ex;
    frexp(a, &ex);  /* a = f * 2^ex, 0.5 <= f < 1 */
    if (ex - 1 > e) e = ex - 1;
  }
  double m = nearbyint(a / ldexp(1.0, e - 3));  /* exact quotient; ties to even */
  int code = 8 * (e + 6) + (int)m;
  if (code > 0x7e) code = 0x7e;
  return sign | (uint8_t)code;
}

/* Element offset of (logical position j, kv head g, dim 0) of sequence s. */
static int64_t cache_offset(const int32_t *block_table, int max_pages, int s,
                            int64_t j, int g, int Hkv, int D, int page_size) {
  int64_t page = block_table[(int64_t)s * max_pages + j / page_size];
  int64_t off = j % page_size;
  return ((page * Hkv + g) * page_size + off) * (int64_t)D;
}

typedef struct {
  const void *q, *k_cache, *v_cache;
  int dtype;     /* element type of q */
  int kv_dtype;  /* element type of the caches */
  double k_scale, v_scale;  /* cache values are stored values times these */
  const int32_t *block_table;
  int max_pages;
  const int32_t *query_start_loc, *seq_lens;
  int num_seqs, Hq, Hkv, D, page_size;
  double scale;
} oracle_problem;

/* Sequence that owns packed query token t (linear scan; plain on purpose). */
static int owner_seq(const oracle_problem *P, int64_t t) {
  for (int s = 0; s < P->num_seqs; ++s)
    if (t >= P->query_start_loc[s] && t < P->query_start_loc[s + 1]) return s;
  return -1;
}

/* Attention of one (query token t, head h).  Writes D doubles to out and, if
 * probs is not NULL, the ctx-q_len+i+1 softmax weights.  Returns the number of
 * visible keys, or -1 on malformed metadata. */
static int64_t attend_one(const oracle_problem *P, int64_t t, int h,
                          double *out, double *probs, double *scratch) {
  int s = owner_seq(P, t);
  if (s < 0) return -1;
  int64_t q_len = P->query_start_loc[s + 1] - P->query_start_loc[s];
  int64_t ctx = P->seq_lens[s];
  int64_t i = t - P->query_start_loc[s];
  if (ctx < q_len) return -1;
  int64_t last = ctx - q_len + i;              /* last visible key */
  int64_t n_vis = last + 1;
  int g = h / (P->Hq / P->Hkv);                /* GQA: contiguous groups */
  int D = P->D;
  int64_t q_base = (t * P->Hq + h) * (int64_t)D;

  double *x = scratch;                         /* n_vis logits */
  double mx = -INFINITY;
  for (int64_t j = 0; j < n_vis; ++j) {
    int64_t kb = cache_offset(P->block_table, P->max_pages, s, j, g, P->Hkv, D,
                              P->page_size);
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += load_elem(P->q, P->dtype, q_base + d) *
             load_elem(P->k_cache, P->kv_dtype, kb + d);
    dot *= P->k_scale;                         /* K = k_scale * stored K */
    x[j] = P->scale * dot;
    if (x[j] > mx) mx = x[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n_vis; ++j) {
    x[j] = exp(x[j] - mx);
    z += x[j];
  }
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int64_t j = 0; j < n_vis; ++j) {
    double p = x[j] / z;
    if (probs) probs[j] = p;
    int64_t vb = cache_offset(P->block_table, P->max_pages, s, j, g, P->Hkv, D,
                              P->page_size);
    double pv = p * P->v_scale;                /* V = v_scale * stored V */
    for (int d = 0; d < D; ++d) out[d] += pv * load_elem(P->v_cache, P->kv_dtype, vb + d);
  }
  return n_vis;
}

typedef struct {
  const oracle_problem *P;
  const int64_t *rows;   /* packed token indices to evaluate */
  int64_t first, count;  /* this worker's slice of rows[] */
  double *out;           /* [num_rows][Hq][D] */
  int64_t max_ctx;
  int status;
} oracle_job;

static void *run_job(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  const oracle_problem *P = J->P;
  double *scratch = (double *)malloc(sizeof(double) * (size_t)(J->max_ctx + 1));
  if (!scratch) { J->status = -2; return NULL; }
  for (int64_t r = J->first; r < J->first + J->count; ++r) {
    for (int h = 0; h < P->Hq; ++h) {
      double *o = J->out + (r * P->Hq + h) * (int64_t)P->D;
      if (attend_one(P, J->rows[r], h, o, NULL, scratch) < 0) J->status = -1;
    }
  }
  free(scratch);
  return NULL;
}

/* Attention output for the packed query tokens listed in rows[0..num_rows),
 * q of element type q_dtype, caches of element type kv_dtype holding
 * K / k_scale and V / v_scale.  out is [num_rows][Hq][D] doubles.
 * nthreads >= 1 workers split the rows.  Returns 0, or -1 on malformed
 * metadata, -2 on allocation failure. */
int oracle_attention_kv(const void *q, int q_dtype, const void *k_cache,
                        const void *v_cache, int kv_dtype, double k_scale,
                        double v_scale, const int32_t *block_table, int max_pages,
                        const int32_t *query_start_loc, const int32_t *seq_lens,
                        int num_seqs, int Hq, int Hkv, int D, int page_size,
                        double scale, const int64_t *rows, int64_t num_rows,
                        double *out, int nthreads) {
  if (Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0 || D <= 0) return -1;
  oracle_problem P = {q, k_cache, v_cache, q_dtype, kv_dtype, k_scale, v_scale,
                      block_table, max_pages, query_start_loc, seq_lens,
                      num_seqs, Hq, Hkv, D, page_size, scale};
  int64_t max_ctx = 0;
  for (int s = 0; s < num_seqs; ++s)
    if (seq_lens[s] > max_ctx) max_ctx = seq_lens[s];
  if (nthreads < 1) nthreads = 1;
  if (nthreads > num_rows) nthreads = num_rows > 0 ? (int)num_rows : 1;
  oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) { free(jobs); free(tids); return -2; }
  int64_t per = num_rows / nthreads, extra = num_rows % nthreads, first = 0;
  for (int w = 0; w < nthreads; ++w) {
    int64_t cnt = per + (w < extra ? 1 : 0);
    jobs[w] = (oracle_job){&P, rows, first, cnt, out, max_ctx, 0};
    first += cnt;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tids[w], NULL, run_job, &jobs[w]);
  run_job(&jobs[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tids[w], NULL);
  int status = 0;
  for (int w = 0; w < nthreads; ++w)
    if (jobs[w].status) status = jobs[w].status;
  free(jobs);
  free(tids);
  return status;
}

/* The same with q and caches of one element type and unit scales. */
int oracle_attention(const void *q, const void *k_cache, const void *v_cache,
                     int dtype, const int32_t *block_table, int max_pages,
                     const int32_t *query_start_loc, const int32_t *seq_lens,
                     int num_seqs, int Hq, int Hkv, int D, int page_size,
                     double scale, const int64_t *rows, int64_t num_rows,
                     double *out, int nthreads) {
  return oracle_attention_kv(q, dtype, k_cache, v_cache, dtype, 1.0, 1.0,
                             block_table, max_pages, query_start_loc, seq_lens,
                             num_seqs, Hq, Hkv, D, page_size, scale, rows,
                             num_rows, out, nthreads);
}

/* Softmax weights of one (packed token t, head h) over its visible keys.
 * probs must hold seq_lens[s] doubles; out holds D doubles.  Returns the
 * number of visible keys, or a negative status. */
int64_t oracle_probs(const void *q, const void *k_cache, const void *v_cache,
                     int dtype, const int32_t *block_table, int max_pages,
                     const int32_t *query_start_loc, const int32_t *seq_lens,
                     int num_seqs, int Hq, int Hkv, int D, int page_size,
                     double scale, int64_t t, int h, double *probs, double *out) {
  if (Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0 || D <= 0) return -1;
  oracle_problem P = {q, k_cache, v_cache, dtype, dtype, 1.0, 1.0, block_table,
                      max_pages, query_start_loc, seq_lens, num_seqs, Hq, Hkv,
                      D, page_size, scale};
  int s = owner_seq(&P, t);
  if (s < 0) return -1;
  double *scratch = (double *)malloc(sizeof(double) * (size_t)(seq_lens[s] + 1));
  if (!scratch) return -2;
  int64_t n = attend_one(&P, t, h, out, probs, scratch);
  free(scratch);
  return n;
}

/* KV append: copy token t's K and V rows (all kv heads) into cache slot
 * slot_mapping[t]; a negative slot means "no cache write".  A slot is
 * page * page_size + offset.  Bytes are copied verbatim, so the result is the
 * bit pattern of the inputs ("Chunked Prefill on an M5 Max", section "Wiring it
 * into the loop": a chunk extends the cache rather than rebuilding it). */
void oracle_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                      int64_t num_tokens, int Hkv, int D, int page_size,
                      int elem_bytes, void *k_cache, void *v_cache) {
  size_t row = (size_t)D * (size_t)elem_bytes;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t page = slot / page_size, off = slot % page_size;
    for (int g = 0; g < Hkv; ++g) {
      size_t dst = (size_t)(((page * Hkv + g) * page_size + off)) * row;
      size_t src = (size_t)(t * Hkv + g) * row;
      memcpy((char *)k_cache + dst, (const char *)k + src, row);
      memcpy((char *)v_cache + dst, (const char *)v + src, row);
    }
  }
}

/* E4M3 codes of x[0..n) / scale, the quotient taken in binary32 (one
 * correctly rounded division), x of element type dtype. */
void oracle_e4m3_encode(const void *x, int dtype, int64_t n, float scale,
                        uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) {
    float xi = (float)load_elem(x, dtype, i);  /* exact: every input type fits */
    float y = xi / scale;
    out[i] = e4m3_code(y);
  }
}

/* Values of E4M3 codes. */
void oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

/* Values of IEEE binary16 bit patterns. */
void oracle_f16_decode(const uint16_t *bits, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_value(bits[i]);
}

/* KV append into an E4M3 cache: token t's K row (all kv heads) is stored as
 * the codes of k / k_scale at slot_mapping[t], V likewise with v_scale; a
 * negative slot means "no cache write".  k and v have element type dtype. */
void oracle_kv_append_e4m3(const void *k, const void *v, int dtype,
                           const int64_t *slot_mapping, int64_t num_tokens,
                           int Hkv, int D, int page_size, float k_scale,
                           float v_scale, uint8_t *k_cache, uint8_t *v_cache) {
  int eb = dtype == ORACLE_F32 ? 4 : 2;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t page = slot / page_size, off = slot % page_size;
    for (int g = 0; g < Hkv; ++g) {
      int64_t dst = ((page * Hkv + g) * page_size + off) * (int64_t)D;
      int64_t src = (t * Hkv + g) * (int64_t)D;
      oracle_e4m3_encode((const char *)k + src * eb, dtype, D, k_scale, k_cache + dst);
      oracle_e4m3_encode((const char *)v + src * eb, dtype, D, v_scale, v_cache + dst);
    }
  }
}

/* Cache slot of every new token of the step: the q_len new tokens of sequence
 * s sit at logical positions ctx-q_len .. ctx-1 ("Chunked Prefill 技术深度解析",
 * section 4.2: pages of 16 tokens, found through the request's page list). */
int oracle_slot_mapping(const int32_t *block_table, int max_pages,
                        const int32_t *query_start_loc, const int32_t *seq_lens,
                        int num_seqs, int page_size, int64_t *slot_out) {
  for (int s = 0; s < num_seqs; ++s) {
    int64_t q_len = query_start_loc[s + 1] - query_start_loc[s];
    int64_t ctx = seq_lens[s];
    if (q_len < 0 || ctx < q_len) return -1;
    for (int64_t i = 0; i < q_len; ++i) {
      int64_t pos = ctx - q_len + i;
      int64_t page = block_table[(int64_t)s * max_pages + pos / page_size];
      slot_out[query_start_loc[s] + i] = page * page_size + pos % page_size;
    }
  }
  return 0;
}
