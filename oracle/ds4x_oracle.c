/*
 * ds4x_oracle.c — plain, slow, obviously-correct CPU oracle of the lightning-indexer
 * path.  TEST INFRASTRUCTURE ONLY: it exists to check the CUDA library and is called
 * only by the tests, the smoke check and the benchmark's CPU-baseline leg.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Every floating-point step is done in IEEE double and rounded once at the end.
 * Argument order mirrors the C ABI (include/ds4x.h) but every pointer is a HOST pointer.
 *
 * What it follows:
 *  - Scoring and the top-512 selection: "How I made DeepSeek 12x faster on a Mac
 *    Studio", section "1: the kernels" (the lightning indexer scores compressed KV and
 *    keeps the top 512 rows per token; the streaming top-k of #832 is byte-identical to
 *    a full sort, so the selection is the exact, deterministic one computed here by a
 *    full sort).
 *  - The shortcut: "How I turned one oversized DeepSeek optimization into three merged
 *    oMLX PRs", section "The three changes that merged", item 3: when every pooled row
 *    fits inside index_topk nothing can be eliminated, scoring is skipped and the
 *    sequential indices are built directly.
 *  - A CPU path kept only to verify accuracy: the ds4.c overview (id.news.hada.io,
 *    sections "Gambaran proyek dan filosofi desain" and "Backend").
 *  - The decode loop: one pooled row per `ratio` positions ("How I turned one oversized
 *    DeepSeek optimization into three merged oMLX PRs", section "The three changes that
 *    merged"), decode at long context ("How I made DeepSeek 12x faster on a Mac Studio").
 *  - Local-plus-pooled attention: "How I turned one oversized DeepSeek optimization into
 *    three merged oMLX PRs", section "The three changes that merged", item 1 (compressed
 *    attention draws on local and pooled key/value state; the native kernel takes both in
 *    one pass), and the ds4.c overview, section on the disk cache layout (the live raw
 *    sliding-window KV rows are state of their own).  The pages give no window size and no
 *    rule for joining the two sources; the reading here: the raw rows of the positions
 *    p - window + 1 .. p (none below 0) join the selected pooled rows in one softmax with
 *    the same query and scale, nothing de-duplicated.
 *  - The compressor: one pooled row per `ratio` positions ("three merged oMLX PRs", section
 *    "The three changes that merged", item 3: the skip path still advances the indexer
 *    compressor and its cache), with the partial block carried between calls as state (the
 *    ds4.c overview, disk-cache layout: "compressor frontier" tensors).  The pages give no
 *    formula; the reading here: per channel, a softmax over the block's positions of a gate
 *    logit plus a learned per-position bias weights the block's raw rows (equal gates give the
 *    mean).  Gates, bias and raw rows are inputs (no trained weights exist).
 *  - The formula (which the pages leave unstated) is this library's definition:
 *    score[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]), row s visible iff
 *    (s+1)*ratio <= p+1, ties to the lower row index, indices ascending, attention with
 *    softmax over the selected rows and kv as both key and value.
 *
 * Parity pins (tests/test_oracle.py): brute force in numpy on tiny inputs, an int64
 * recomputation of 4*score on integer inputs, a hand-worked example
 * (tests/golden/indexer_worked_example.txt), the dominance / mask / shortcut
 * invariants of the selection, the closed-form attention cases (zero query ->
 * mean of the rows, one row -> that row, two rows -> logistic weights), and for the
 * decode loop the closed-form row count per step, the appended bytes and a numpy
 * brute-force of every step on tiny inputs; for local-plus-pooled attention a textbook
 * sliding-window attention in numpy, a numpy softmax over the union of both sources, the
 * log-sum-exp merge of the two one-source results, the exact mean for a zero query and a
 * one-row window; for the compressor the exact rational mean under equal gates, a dominant gate
 * giving its row, a numpy softmax pooling, and one call equal to any split into two calls with
 * the frontier carried.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_F16 0
#define REF_BF16 1

/* ---- 16-bit float decoding / encoding, from the IEEE 754 binary16 and the bfloat16
 *      bit layouts (sign | exponent | fraction). ------------------------------------ */

static double ref_f16_to_double(uint16_t h) {
  int sign = h >> 15;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(f + 1024), e - 25);          /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static double ref_bf16_to_double(uint16_t b) {
  int sign = b >> 15;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double v;
  if (e == 0) v = ldexp((double)f, -133);              /* subnormal: f * 2^-133 */
  else if (e == 255) v = f ? NAN : INFINITY;
  else v = ldexp((double)(f + 128), e - 134);          /* (1 + f/128) * 2^(e-127) */
  return sign ? -v : v;
}

static double ref_to_double(uint16_t x, int dtype) {
  return dtype == REF_F16 ? ref_f16_to_double(x) : ref_bf16_to_double(x);
}

/* Round a double to the nearest binary format value with `mant` fraction bits,
 * exponent field width `ebits`, ties to even.  Returns the bit pattern. */
static uint16_t ref_encode(double x, int mant, int ebits) {
  const int bias = (1 << (ebits - 1)) - 1;
  const int emin = 1 - bias;                         /* smallest normal exponent */
  const int emax = bias;                             /* largest normal exponent  */
  uint16_t sign = signbit(x) ? (uint16_t)(1u << (mant + ebits)) : 0;
  uint16_t inf = (uint16_t)(((1u << ebits) - 1) << mant);
  if (isnan(x)) return (uint16_t)(inf | (1u << (mant - 1)));
  double a = fabs(x);
  if (isinf(a)) return sign | inf;
  int e;
  frexp(a, &e);                                      /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;                                     /* a in [2^E, 2^(E+1))        */
  if (a == 0.0 || E < emin) {                        /* subnormal quantum 2^(emin-mant) */
    double r = nearbyint(ldexp(a, mant - emin));     /* default mode: ties to even  */
    /* r == 2^mant rolls over to the smallest normal, which the same packing encodes */
    return sign | (uint16_t)r;
  }
  double r = nearbyint(ldexp(a, mant - E));          /* in [2^mant, 2^(mant+1)]     */
  if (r >= ldexp(1.0, mant + 1)) { r = ldexp(r, -1); E += 1; }
  if (E > emax) return sign | inf;
  return sign | (uint16_t)(((E + bias) << mant) | ((uint32_t)r - (1u << mant)));
}

static uint16_t ref_from_double(double x, int dtype) {
  return dtype == REF_F16 ? ref_encode(x, 10, 5) : ref_encode(x, 7, 8);
}

/* Exposed for the oracle's own pins (exhaustive round trips in the tests). */
double ds4x_ref_decode16(uint16_t x, int dtype) { return ref_to_double(x, dtype); }
uint16_t ds4x_ref_encode16(double x, int dtype) { return ref_from_double(x, dtype); }

/* ---- visibility ------------------------------------------------------------------ */

/* Number of compressed rows visible at position p: row s is visible iff
 * (s+1)*ratio <= p+1, clamped to the S rows that exist. */
int64_t ds4x_ref_n_visible(int64_t p, int64_t ratio, int64_t S) {
  if (p < 0) return 0;
  int64_t n = (p + 1) / ratio;
  return n < S ? n : S;
}

/* ---- scoring ----------------------------------------------------------------------- */

/* Decode n 16-bit values of the given format into doubles (exact). */
static void ref_decode_n(const uint16_t* x, int64_t n, int dtype, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ref_to_double(x[i], dtype);
}

/* One token's scores over rows 0..S-1:
 *   row[s] = (float) sum_h w[h] * max(0, sum_d q[h,d]*k[s,d])   for s < n,
 *   row[s] = -INFINITY                                           for n <= s < S.
 * qd [H*D], wd [H], kd [S*D] are the decoded inputs. */
static void ref_score_token(const double* qd, const double* wd, const double* kd, int64_t n,
                            int32_t H, int32_t D, int64_t S, float* row) {
  for (int64_t s = 0; s < S; ++s) {
    if (s >= n) { row[s] = -INFINITY; continue; }
    const double* ks = kd + s * D;
    double acc = 0.0;
    for (int32_t h = 0; h < H; ++h) {
      const double* qh = qd + (int64_t)h * D;
      double dot = 0.0;
      for (int32_t d = 0; d < D; ++d) dot += qh[d] * ks[d];
      double relu = dot > 0.0 ? dot : 0.0;
      acc += wd[h] * relu;
    }
    row[s] = (float)acc;                               /* one rounding, to nearest even */
  }
}

int ds4x_ref_indexer_score(const uint16_t* q, const uint16_t* w, const uint16_t* k,
                           const int32_t* positions, int32_t T, int32_t H, int32_t D,
                           int32_t S, int32_t ratio, float* scores, int64_t ld_scores) {
  if (T < 0 || H <= 0 || D <= 0 || S < 0 || ratio < 1 || ld_scores < S) return -1;
  double* kd = (double*)malloc(sizeof(double) * (size_t)((int64_t)S * D + 1));
  ref_decode_n(k, (int64_t)S * D, REF_F16, kd);
#pragma omp parallel
  {
    double* qd = (double*)malloc(sizeof(double) * (size_t)H * D);
    double* wd = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
      ref_decode_n(q + (int64_t)t * H * D, (int64_t)H * D, REF_F16, qd);
      ref_decode_n(w + (int64_t)t * H, H, REF_F16, wd);
      int64_t n = ds4x_ref_n_visible(positions[t], ratio, S);
      ref_score_token(qd, wd, kd, n, H, D, S, scores + (int64_t)t * ld_scores);
    }
    free(qd); free(wd);
  }
  free(kd);
  return 0;
}

/* ---- top-k ------------------------------------------------------------------------- */

typedef struct { float score; int32_t idx; } ref_pair;

/* Order used for the selection: higher score first, equal scores -> lower row first. */
static int ref_cmp_pair(const void* a, const void* b) {
  const ref_pair* x = (const ref_pair*)a;
  const ref_pair* y = (const ref_pair*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

static int ref_cmp_int(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Full selection for one token: sort all n visible (score, s) pairs, keep the first
 * k_top, emit them in ascending row order, pad with -1.  Returns the count. */
static int32_t ref_select_one(const float* row, int64_t n, int32_t k_top, int32_t* out) {
  ref_pair* pairs = (ref_pair*)malloc(sizeof(ref_pair) * (size_t)(n > 0 ? n : 1));
  for (int64_t s = 0; s < n; ++s) { pairs[s].score = row[s]; pairs[s].idx = (int32_t)s; }
  qsort(pairs, (size_t)n, sizeof(ref_pair), ref_cmp_pair);
  int32_t c = (int32_t)(n < k_top ? n : k_top);
  for (int32_t i = 0; i < c; ++i) out[i] = pairs[i].idx;
  qsort(out, (size_t)c, sizeof(int32_t), ref_cmp_int);
  for (int32_t i = c; i < k_top; ++i) out[i] = -1;
  free(pairs);
  return c;
}

/* use_shortcut = 1: a token with n_vis <= k_top emits 0..n-1 without reading scores
 * (the oMLX #2563 shortcut).  use_shortcut = 0 runs the full selection for every token
 * (used by the tests to show that both give the same indices). */
int ds4x_ref_topk_ex(const float* scores, int64_t ld_scores, const int32_t* positions,
                     int32_t T, int32_t S, int32_t ratio, int32_t k_top,
                     int32_t* indices, int32_t* counts, int use_shortcut) {
  if (T < 0 || S < 0 || ratio < 1 || k_top < 1 || ld_scores < S) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t t = 0; t < T; ++t) {
    int64_t n = ds4x_ref_n_visible(positions[t], ratio, S);
    int32_t* out = indices + (int64_t)t * k_top;
    int32_t c;
    if (use_shortcut && n <= k_top) {
      for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
      for (int64_t i = n; i < k_top; ++i) out[i] = -1;
      c = (int32_t)n;
    } else {
      c = ref_select_one(scores + (int64_t)t * ld_scores, n, k_top, out);
    }
    if (counts) counts[t] = c;
  }
  return 0;
}

int ds4x_ref_topk(const float* scores, int64_t ld_scores, const int32_t* positions,
                  int32_t T, int32_t S, int32_t ratio, int32_t k_top,
                  int32_t* indices, int32_t* counts) {
  return ds4x_ref_topk_ex(scores, ld_scores, positions, T, S, ratio, k_top, indices, counts, 1);
}

/* ---- sparse multi-query attention -------------------------------------------------- */

/* One token: qd [Hq*Dkv] decoded query, rd [nv*Dkv] decoded selected rows.
 *   l_j = scale * q[h,:] . row_j,  p_j = exp(l_j - max l) / sum exp(l - max l)
 *   out[h,:] = sum_j p_j row_j (rounded once to dtype), lse[h] = max l + log(sum). */
static void ref_attend_token(const double* qd, const double* rd, int32_t nv, int32_t Hq,
                             int32_t Dkv, double scale, int dtype, uint16_t* out, float* lse,
                             double* logit, double* acc) {
  for (int32_t h = 0; h < Hq; ++h) {
    const double* qh = qd + (int64_t)h * Dkv;
    uint16_t* oh = out + (int64_t)h * Dkv;
    if (nv == 0) {
      for (int32_t d = 0; d < Dkv; ++d) oh[d] = ref_from_double(0.0, dtype);
      if (lse) lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int32_t j = 0; j < nv; ++j) {
      const double* r = rd + (int64_t)j * Dkv;
      double dot = 0.0;
      for (int32_t d = 0; d < Dkv; ++d) dot += qh[d] * r[d];
      logit[j] = scale * dot;
      if (logit[j] > m) m = logit[j];
    }
    double sum = 0.0;
    for (int32_t d = 0; d < Dkv; ++d) acc[d] = 0.0;
    for (int32_t j = 0; j < nv; ++j) {
      double p = exp(logit[j] - m);
      sum += p;
      const double* r = rd + (int64_t)j * Dkv;
      for (int32_t d = 0; d < Dkv; ++d) acc[d] += p * r[d];
    }
    for (int32_t d = 0; d < Dkv; ++d) oh[d] = ref_from_double(acc[d] / sum, dtype);
    if (lse) lse[h] = (float)(m + log(sum));
  }
}

/* Attention for every token over its valid selected rows (0 <= idx < S; -1 and
 * out-of-range entries are skipped).  No valid row: out = 0, lse = -inf. */
int ds4x_ref_sparse_attn(const uint16_t* q_attn, const uint16_t* kv, int dtype,
                         const int32_t* indices, int32_t T, int32_t Hq, int32_t Dkv,
                         int32_t S, int32_t k_top, float scale, uint16_t* out, float* lse) {
  if (T < 0 || Hq <= 0 || Dkv <= 0 || S < 0 || k_top < 1) return -1;
#pragma omp parallel
  {
    double* qd = (double*)malloc(sizeof(double) * (size_t)Hq * Dkv);
    double* rd = (double*)malloc(sizeof(double) * (size_t)k_top * Dkv);
    double* logit = (double*)malloc(sizeof(double) * (size_t)k_top);
    double* acc = (double*)malloc(sizeof(double) * (size_t)Dkv);
#pragma omp for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
      const int32_t* sel = indices + (int64_t)t * k_top;
      int32_t nv = 0;
      for (int32_t j = 0; j < k_top; ++j)
        if (sel[j] >= 0 && sel[j] < S)
          ref_decode_n(kv + (int64_t)sel[j] * Dkv, Dkv, dtype, rd + (int64_t)(nv++) * Dkv);
      ref_decode_n(q_attn + (int64_t)t * Hq * Dkv, (int64_t)Hq * Dkv, dtype, qd);
      ref_attend_token(qd, rd, nv, Hq, Dkv, (double)scale, dtype,
                       out + (int64_t)t * Hq * Dkv, lse ? lse + (int64_t)t * Hq : NULL,
                       logit, acc);
    }
    free(qd); free(rd); free(logit); free(acc);
  }
  return 0;
}

/* ---- local-plus-pooled attention ---------------------------------------------------- */

/* The raw rows in a token's sliding window: the positions a with p - window < a <= p and
 * a >= 0 that kv_local holds (its row r is the raw row of position local_pos0 + r, r < L),
 * in ascending position.  Writes their kv_local row numbers and returns how many. */
static int32_t ref_window_rows(int64_t p, int32_t window, int64_t local_pos0, int32_t L,
                               int32_t* rows) {
  int32_t n = 0;
  for (int64_t a = p - window + 1; a <= p; ++a) {
    if (a < 0) continue;
    int64_t r = a - local_pos0;
    if (r < 0 || r >= L) continue;
    rows[n++] = (int32_t)r;
  }
  return n;
}

/* One softmax over two row sources: the token's valid selected pooled rows (as in
 * ds4x_ref_sparse_attn) followed by the raw rows of its sliding window.  Both sources are
 * keys and values; the logits share q_attn and scale.  window = 0 or L = 0 gives
 * ds4x_ref_sparse_attn. */
int ds4x_ref_local_pooled_attn(const uint16_t* q_attn, const uint16_t* kv,
                               const uint16_t* kv_local, int dtype, const int32_t* indices,
                               const int32_t* positions, int32_t T, int32_t Hq, int32_t Dkv,
                               int32_t S, int32_t k_top, int32_t local_pos0, int32_t L,
                               int32_t window, float scale, uint16_t* out, float* lse) {
  if (T < 0 || Hq <= 0 || Dkv <= 0 || S < 0 || k_top < 1 || L < 0 || window < 0 || local_pos0 < 0)
    return -1;
  const int64_t cap = (int64_t)k_top + window;
#pragma omp parallel
  {
    double* qd = (double*)malloc(sizeof(double) * (size_t)Hq * Dkv);
    double* rd = (double*)malloc(sizeof(double) * (size_t)cap * Dkv);
    double* logit = (double*)malloc(sizeof(double) * (size_t)cap);
    double* acc = (double*)malloc(sizeof(double) * (size_t)Dkv);
    int32_t* wrows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(window > 0 ? window : 1));
#pragma omp for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
      const int32_t* sel = indices + (int64_t)t * k_top;
      int32_t nv = 0;
      for (int32_t j = 0; j < k_top; ++j)
        if (sel[j] >= 0 && sel[j] < S)
          ref_decode_n(kv + (int64_t)sel[j] * Dkv, Dkv, dtype, rd + (int64_t)(nv++) * Dkv);
      const int32_t nw = ref_window_rows(positions[t], window, local_pos0, L, wrows);
      for (int32_t j = 0; j < nw; ++j)
        ref_decode_n(kv_local + (int64_t)wrows[j] * Dkv, Dkv, dtype, rd + (int64_t)(nv++) * Dkv);
      ref_decode_n(q_attn + (int64_t)t * Hq * Dkv, (int64_t)Hq * Dkv, dtype, qd);
      ref_attend_token(qd, rd, nv, Hq, Dkv, (double)scale, dtype,
                       out + (int64_t)t * Hq * Dkv, lse ? lse + (int64_t)t * Hq : NULL,
                       logit, acc);
    }
    free(qd); free(rd); free(logit); free(acc); free(wrows);
  }
  return 0;
}

/* ---- the whole path ----------------------------------------------------------------- */

/* score -> top-k (with the shortcut): the indices of every token.  A token covered by the
 * shortcut (n_vis <= k_top) is never scored. */
static void ref_index_select(const uint16_t* q, const uint16_t* w, const uint16_t* k,
                             const int32_t* positions, int32_t T, int32_t H, int32_t D,
                             int32_t S, int32_t ratio, int32_t k_top, int32_t* indices) {
  double* kd = (double*)malloc(sizeof(double) * (size_t)((int64_t)S * D + 1));
  ref_decode_n(k, (int64_t)S * D, REF_F16, kd);
#pragma omp parallel
  {
    double* qd = (double*)malloc(sizeof(double) * (size_t)H * D);
    double* wd = (double*)malloc(sizeof(double) * (size_t)H);
    float* row = (float*)malloc(sizeof(float) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
      int64_t n = ds4x_ref_n_visible(positions[t], ratio, S);
      int32_t* sel = indices + (int64_t)t * k_top;
      if (n <= k_top) {                                  /* shortcut: nothing to rank */
        for (int64_t i = 0; i < k_top; ++i) sel[i] = i < n ? (int32_t)i : -1;
        continue;
      }
      ref_decode_n(q + (int64_t)t * H * D, (int64_t)H * D, REF_F16, qd);
      ref_decode_n(w + (int64_t)t * H, H, REF_F16, wd);
      ref_score_token(qd, wd, kd, n, H, D, S, row);
      ref_select_one(row, n, k_top, sel);
    }
    free(qd); free(wd); free(row);
  }
  free(kd);
}

/* score -> top-k (with the shortcut) -> attention. */
int ds4x_ref_index_and_attend(const uint16_t* q, const uint16_t* w, const uint16_t* k,
                              const int32_t* positions, const uint16_t* q_attn,
                              const uint16_t* kv, int kv_dtype, int32_t T, int32_t H,
                              int32_t D, int32_t S, int32_t ratio, int32_t k_top,
                              int32_t Hq, int32_t Dkv, float scale, int32_t* indices,
                              uint16_t* out, float* lse) {
  if (T < 0 || H <= 0 || D <= 0 || S < 0 || ratio < 1 || k_top < 1) return -1;
  ref_index_select(q, w, k, positions, T, H, D, S, ratio, k_top, indices);
  return ds4x_ref_sparse_attn(q_attn, kv, kv_dtype, indices, T, Hq, Dkv, S, k_top, scale, out, lse);
}

/* score -> top-k (with the shortcut) -> local-plus-pooled attention. */
int ds4x_ref_index_and_attend_local(const uint16_t* q, const uint16_t* w, const uint16_t* k,
                                    const int32_t* positions, const uint16_t* q_attn,
                                    const uint16_t* kv, const uint16_t* kv_local, int kv_dtype,
                                    int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio,
                                    int32_t k_top, int32_t Hq, int32_t Dkv, int32_t local_pos0,
                                    int32_t L, int32_t window, float scale, int32_t* indices,
                                    uint16_t* out, float* lse) {
  if (T < 0 || H <= 0 || D <= 0 || S < 0 || ratio < 1 || k_top < 1 || L < 0 || window < 0)
    return -1;
  ref_index_select(q, w, k, positions, T, H, D, S, ratio, k_top, indices);
  return ds4x_ref_local_pooled_attn(q_attn, kv, kv_local, kv_dtype, indices, positions, T, Hq,
                                    Dkv, S, k_top, local_pos0, L, window, scale, out, lse);
}

/* ---- the compressor ------------------------------------------------------------------ */

/* Row v of the sequence made of the n_frontier held-over positions followed by the T new ones. */
static const uint16_t* ref_seq_row(const uint16_t* held, const uint16_t* fresh, int32_t n_frontier,
                                   int64_t v, int32_t D) {
  return v < n_frontier ? held + v * D : fresh + (v - n_frontier) * D;
}

/* One compressed row per `ratio` consecutive positions.  The sequence is the n_frontier
 * positions held over from the previous call (fx_in, fg_in) followed by the T new positions
 * (x, g).  Block j covers sequence positions j*ratio .. j*ratio + ratio - 1 and gives, per
 * channel d, with i the position inside the block:
 *   rows[j,d] = sum_i a_i x_i[d],   a_i = exp(z_i) / sum_i' exp(z_i'),   z_i = g_i[d] + bias[i,d]
 * (max-subtracted, in double, rounded once to dtype).  The (n_frontier + T) mod ratio positions
 * after the last full block are copied to fx_out / fg_out: the new frontier. */
int ds4x_ref_compress(const uint16_t* x, const uint16_t* g, const float* bias, int dtype,
                      int32_t T, int32_t D, int32_t ratio, const uint16_t* fx_in,
                      const uint16_t* fg_in, int32_t n_frontier, uint16_t* rows,
                      uint16_t* fx_out, uint16_t* fg_out) {
  if (T < 0 || D < 1 || ratio < 1 || n_frontier < 0 || n_frontier >= ratio) return -1;
  const int64_t n = (int64_t)n_frontier + T;
  const int64_t n_out = n / ratio;
  double* z = (double*)malloc(sizeof(double) * (size_t)ratio);
  for (int64_t j = 0; j < n_out; ++j) {
    for (int32_t d = 0; d < D; ++d) {
      double m = -INFINITY;
      for (int32_t i = 0; i < ratio; ++i) {
        const int64_t v = j * ratio + i;
        z[i] = ref_to_double(ref_seq_row(fg_in, g, n_frontier, v, D)[d], dtype) +
               (double)bias[(int64_t)i * D + d];
        if (z[i] > m) m = z[i];
      }
      double sum = 0.0, acc = 0.0;
      for (int32_t i = 0; i < ratio; ++i) {
        const int64_t v = j * ratio + i;
        const double a = exp(z[i] - m);
        sum += a;
        acc += a * ref_to_double(ref_seq_row(fx_in, x, n_frontier, v, D)[d], dtype);
      }
      rows[j * D + d] = ref_from_double(acc / sum, dtype);
    }
  }
  for (int64_t v = n_out * ratio; v < n; ++v) {
    const int64_t i = v - n_out * ratio;
    memcpy(fx_out + i * D, ref_seq_row(fx_in, x, n_frontier, v, D), sizeof(uint16_t) * (size_t)D);
    memcpy(fg_out + i * D, ref_seq_row(fg_in, g, n_frontier, v, D), sizeof(uint16_t) * (size_t)D);
  }
  free(z);
  return 0;
}

/* ---- the decode loop ------------------------------------------------------------------ */

/* n_steps single-token steps at positions p = pos0 + i.  Before step i, while S is below the
 * number of rows p may see (floor((p+1)/ratio)) and a staged row and capacity are left, the
 * next staged row (k_new[a], kv_new[a]) is copied to row S of k and kv and S grows by one.
 * Step i is then ds4x_ref_index_and_attend for that one token with the current S; S_steps[i]
 * records that S.  k and kv are host arrays of `capacity` rows, updated in place. */
int ds4x_ref_decode(const uint16_t* q, const uint16_t* w, const uint16_t* q_attn, uint16_t* k,
                    uint16_t* kv, int kv_dtype, int32_t capacity, int32_t S0,
                    const uint16_t* k_new, const uint16_t* kv_new, int32_t n_new, int32_t pos0,
                    int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top,
                    int32_t Hq, int32_t Dkv, float scale, int32_t* positions, int32_t* indices,
                    uint16_t* out, float* lse, int32_t* S_steps) {
  if (n_steps < 0 || capacity < 1 || S0 < 0 || S0 > capacity || n_new < 0 || ratio < 1 || pos0 < 0)
    return -1;
  int32_t S = S0, a = 0;
  for (int32_t i = 0; i < n_steps; ++i) {
    const int64_t p = (int64_t)pos0 + i;
    positions[i] = (int32_t)p;
    while (S < capacity && a < n_new && (int64_t)S < (p + 1) / ratio) {
      memcpy(k + (int64_t)S * D, k_new + (int64_t)a * D, sizeof(uint16_t) * (size_t)D);
      memcpy(kv + (int64_t)S * Dkv, kv_new + (int64_t)a * Dkv, sizeof(uint16_t) * (size_t)Dkv);
      ++S;
      ++a;
    }
    S_steps[i] = S;
    int rc = ds4x_ref_index_and_attend(q + (int64_t)i * H * D, w + (int64_t)i * H, k, positions + i,
                                       q_attn + (int64_t)i * Hq * Dkv, kv, kv_dtype, 1, H, D, S, ratio,
                                       k_top, Hq, Dkv, scale, indices + (int64_t)i * k_top,
                                       out + (int64_t)i * Hq * Dkv, lse + (int64_t)i * Hq);
    if (rc != 0) return rc;
  }
  return 0;
}

/* The decode loop with local-plus-pooled attention: as ds4x_ref_decode, and before the first step
 * the n_steps raw rows kv_raw_new land at rows pos0 .. pos0 + n_steps - 1 of kv_raw (row a = the
 * raw row of position a; rows below pos0 are the caller's history); step i (position p) is
 * ds4x_ref_index_and_attend_local over kv_raw with the window.  kv_raw holds raw_capacity rows
 * (>= pos0 + n_steps) and is updated in place. */
int ds4x_ref_decode_local(const uint16_t* q, const uint16_t* w, const uint16_t* q_attn, uint16_t* k,
                          uint16_t* kv, int kv_dtype, int32_t capacity, int32_t S0,
                          const uint16_t* k_new, const uint16_t* kv_new, int32_t n_new, int32_t pos0,
                          int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top,
                          int32_t Hq, int32_t Dkv, float scale, uint16_t* kv_raw,
                          int32_t raw_capacity, const uint16_t* kv_raw_new, int32_t window,
                          int32_t* positions, int32_t* indices, uint16_t* out, float* lse,
                          int32_t* S_steps) {
  if (n_steps < 0 || capacity < 1 || S0 < 0 || S0 > capacity || n_new < 0 || ratio < 1 || pos0 < 0 ||
      window < 0 || (int64_t)pos0 + n_steps > raw_capacity)
    return -1;
  memcpy(kv_raw + (int64_t)pos0 * Dkv, kv_raw_new, sizeof(uint16_t) * (size_t)n_steps * Dkv);
  int32_t S = S0, a = 0;
  for (int32_t i = 0; i < n_steps; ++i) {
    const int64_t p = (int64_t)pos0 + i;
    positions[i] = (int32_t)p;
    while (S < capacity && a < n_new && (int64_t)S < (p + 1) / ratio) {
      memcpy(k + (int64_t)S * D, k_new + (int64_t)a * D, sizeof(uint16_t) * (size_t)D);
      memcpy(kv + (int64_t)S * Dkv, kv_new + (int64_t)a * Dkv, sizeof(uint16_t) * (size_t)Dkv);
      ++S;
      ++a;
    }
    S_steps[i] = S;
    int rc = ds4x_ref_index_and_attend_local(q + (int64_t)i * H * D, w + (int64_t)i * H, k, positions + i,
                                             q_attn + (int64_t)i * Hq * Dkv, kv, kv_raw, kv_dtype, 1, H, D, S,
                                             ratio, k_top, Hq, Dkv, 0, pos0 + n_steps, window, scale,
                                             indices + (int64_t)i * k_top, out + (int64_t)i * Hq * Dkv,
                                             lse + (int64_t)i * Hq);
    if (rc != 0) return rc;
  }
  return 0;
}

