/*
 * oracle.c -- plain, slow fp64 CPU oracle for the predictive sparse-KV decode
 * step ("DualDecoder: Accelerate Long Context LLM Inference by Predictive
 * Prefetch", arXiv:2607.26475).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code
 * with the CUDA path (no headers, helpers, tables or constants).
 *
 * What it computes, per layer and per (request b, KV head h_kv):
 *   1. logits   s_h[j] = (q_spec[h] . K[j]) / sqrt(d_k) for every query head h
 *               of the group and every cached position j < n
 *               (paper summary page, "core formulas": alpha = softmax(q_spec K^T /
 *               sqrt(d_k)); the worked example scales by the square root of
 *               the per-head key size);
 *   2. softmax  LSE_h = log sum_j exp(s_h[j]), alpha_h[j] = exp(s_h[j] - LSE_h)
 *               (same formula);
 *   3. score    a[j] = alpha_h[j] for MHA, a[j] = sum_{h in group} alpha_h[j]
 *               for grouped-query heads (one selection per KV head);
 *   4. select   I = argtopk(a, k) over j in [0, n - W): sort by (a desc, j asc),
 *               keep the first k, report them in ascending j (same formula;
 *               paper Fig. 1 "Select Top-k"); ties go to the lower index;
 *   5. attend   o_h = sum_{j in S} softmax_S(q[h] . K[j] / sqrt(d)) V[j] over
 *               S = I  union  [n - W, n)  (paper Fig. 1 "Attention" over the
 *               gathered sparse KV; summary page worked example, step 6);
 *   6. dense    the same as 5 with S = [0, n) (paper Sec. 2.1: attention of
 *               the current query over all cached KV entries).
 * Every input is the exact stored value (bf16 or fp32) widened to double.
 * Parity of every function here is pinned by the tests against closed forms,
 * invariants and brute force, not against this file.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

typedef struct {
  int32_t batch, n_q_heads, n_kv_heads, head_dim, ctx_len, top_k, window, dtype;
} orc_shape;

/* Stored element i of a bf16 (upper 16 bits of an IEEE binary32) or fp32 array. */
static double widen(const void* p, int dtype, int64_t i) {
  float f;
  if (dtype == ORC_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    memcpy(&f, &bits, 4);
  } else {
    f = ((const float*)p)[i];
  }
  return (double)f;
}

static int group_size(const orc_shape* s) { return s->n_q_heads / s->n_kv_heads; }

/* q[b][h][:] . X[b][h_kv][j][:] in fp64 (q is [B][H_q][d], X is [B][H_kv][n][d]). */
static double dot_row(const orc_shape* s, const void* q, int64_t q_off, const void* X, int64_t x_off) {
  double acc = 0.0;
  for (int t = 0; t < s->head_dim; ++t)
    acc += widen(q, s->dtype, q_off + t) * widen(X, s->dtype, x_off + t);
  return acc;
}

/*
 * Steps 1-2 for unit (b, hk).  logits is [G][n], lse is [G].
 * LSE_h = m + log sum_j exp(s_h[j] - m), m = max_j s_h[j]  (textbook
 * log-sum-exp; the shift by m only avoids overflow).
 */
void orc_score_unit(const orc_shape* s, const void* q_spec, const void* K, int b, int hk,
                    double* logits, double* lse) {
  const int G = group_size(s), d = s->head_dim, n = s->ctx_len;
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  for (int g = 0; g < G; ++g) {
    const int h = hk * G + g;
    const int64_t q_off = ((int64_t)b * s->n_q_heads + h) * d;
    double* lg = logits + (int64_t)g * n;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      const int64_t k_off = (((int64_t)b * s->n_kv_heads + hk) * n + j) * d;
      lg[j] = dot_row(s, q_spec, q_off, K, k_off) * inv_sqrt_d;
      if (lg[j] > m) m = lg[j];
    }
    double sum = 0.0;
    for (int j = 0; j < n; ++j) sum += exp(lg[j] - m);
    lse[g] = m + log(sum);
  }
}

/* Step 3: a[j] = sum over the group of alpha_h[j] = exp(s_h[j] - LSE_h). */
void orc_selection_score(const orc_shape* s, const double* logits, const double* lse, double* a) {
  const int G = group_size(s), n = s->ctx_len;
  for (int j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int g = 0; g < G; ++g) acc += exp(logits[(int64_t)g * n + j] - lse[g]);
    a[j] = acc;
  }
}

typedef struct {
  double a;
  int32_t j;
} cand;

/* (a desc, j asc): the strict total order that breaks ties toward lower j. */
static int by_score_desc(const void* x, const void* y) {
  const cand* p = (const cand*)x;
  const cand* q = (const cand*)y;
  if (p->a > q->a) return -1;
  if (p->a < q->a) return 1;
  return (p->j < q->j) ? -1 : (p->j > q->j);
}

static int by_index_asc(const void* x, const void* y) {
  const cand* p = (const cand*)x;
  const cand* q = (const cand*)y;
  return (p->j < q->j) ? -1 : (p->j > q->j);
}

/*
 * Step 4 for one unit: a is [n] (step 3).  Writes idx[k] (ascending j) and
 * sel[k] = a[idx].  *gap = (a_(k) - a_(k+1)) / a_(k), the relative gap
 * between the k-th and (k+1)-th largest score in the order above
 * (+inf when k == n - W: nothing is left out).
 */
void orc_select_unit(const orc_shape* s, const double* a, int32_t* idx, double* sel, double* gap) {
  const int span = s->ctx_len - s->window, k = s->top_k;
  cand* c = (cand*)malloc(sizeof(cand) * (size_t)span);
  for (int j = 0; j < span; ++j) {
    c[j].a = a[j];
    c[j].j = j;
  }
  qsort(c, (size_t)span, sizeof(cand), by_score_desc);
  if (gap) *gap = (k < span) ? (c[k - 1].a - c[k].a) / c[k - 1].a : INFINITY;
  qsort(c, (size_t)k, sizeof(cand), by_index_asc);
  for (int i = 0; i < k; ++i) {
    idx[i] = c[i].j;
    if (sel) sel[i] = c[i].a;
  }
  free(c);
}

/*
 * Step 5 for unit (b, hk): softmax attention of the real query q over the
 * positions idx[0..n_idx) followed, if include_window, by [n - W, n).
 * out is [G][d].  K, V are [B][H_kv][n][d]; q is [B][H_q][d].
 */
void orc_attend_unit(const orc_shape* s, const void* q, const void* K, const void* V, int b, int hk,
                     const int32_t* idx, int64_t n_idx, int include_window, double* out) {
  const int G = group_size(s), d = s->head_dim, n = s->ctx_len;
  const int64_t n_win = include_window ? s->window : 0;
  const int64_t m_rows = n_idx + n_win;
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  const int64_t unit_row0 = ((int64_t)b * s->n_kv_heads + hk) * n;
  double* e = (double*)malloc(sizeof(double) * (size_t)(m_rows > 0 ? m_rows : 1));
  for (int g = 0; g < G; ++g) {
    const int h = hk * G + g;
    const int64_t q_off = ((int64_t)b * s->n_q_heads + h) * d;
    double m = -INFINITY;
    for (int64_t r = 0; r < m_rows; ++r) {
      const int64_t j = (r < n_idx) ? idx[r] : (n - n_win + (r - n_idx));
      e[r] = dot_row(s, q, q_off, K, (unit_row0 + j) * d) * inv_sqrt_d;
      if (e[r] > m) m = e[r];
    }
    double z = 0.0;
    for (int64_t r = 0; r < m_rows; ++r) z += exp(e[r] - m);
    double* o = out + (int64_t)g * d;
    for (int t = 0; t < d; ++t) o[t] = 0.0;
    for (int64_t r = 0; r < m_rows; ++r) {
      const int64_t j = (r < n_idx) ? idx[r] : (n - n_win + (r - n_idx));
      const double p = exp(e[r] - m) / z;
      for (int t = 0; t < d; ++t) o[t] += p * widen(V, s->dtype, (unit_row0 + j) * d + t);
    }
  }
  free(e);
}

/* Step 6: dense softmax attention over every cached position [0, n). */
void orc_dense_unit(const orc_shape* s, const void* q, const void* K, const void* V, int b, int hk,
                    double* out) {
  int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)s->ctx_len);
  for (int j = 0; j < s->ctx_len; ++j) all[j] = j;
  orc_attend_unit(s, q, K, V, b, hk, all, s->ctx_len, 0, out);
  free(all);
}

/* ---------------- whole layer: steps 1-5 over every unit ---------------- */

typedef struct {
  const orc_shape* s;
  const void *q_spec, *q, *K, *V;
  int32_t* idx;   /* [B][H_kv][k] */
  double* sel;    /* [B][H_kv][k] */
  double* lse;    /* [B][H_q] */
  double* gap;    /* [B][H_kv] */
  double* out;    /* [B][H_q][d] */
  int64_t lo, hi; /* unit range */
} layer_job;

static void* layer_worker(void* p) {
  layer_job* J = (layer_job*)p;
  const orc_shape* s = J->s;
  const int G = group_size(s), n = s->ctx_len, k = s->top_k, d = s->head_dim;
  double* logits = (double*)malloc(sizeof(double) * (size_t)G * n);
  double* a = (double*)malloc(sizeof(double) * (size_t)n);
  for (int64_t u = J->lo; u < J->hi; ++u) {
    const int b = (int)(u / s->n_kv_heads), hk = (int)(u % s->n_kv_heads);
    double* lse = J->lse + ((int64_t)b * s->n_q_heads + (int64_t)hk * G);
    orc_score_unit(s, J->q_spec, J->K, b, hk, logits, lse);
    orc_selection_score(s, logits, lse, a);
    orc_select_unit(s, a, J->idx + u * k, J->sel + u * k, J->gap + u);
    orc_attend_unit(s, J->q, J->K, J->V, b, hk, J->idx + u * k, k, 1,
                    J->out + ((int64_t)b * s->n_q_heads + (int64_t)hk * G) * d);
  }
  free(logits);
  free(a);
  return NULL;
}

/* Steps 1-5 for units [u_lo, u_hi) of a layer, split over nthreads threads. */
void orc_layer(const orc_shape* s, const void* q_spec, const void* q, const void* K, const void* V,
               int32_t* idx, double* sel, double* lse, double* gap, double* out, int64_t u_lo,
               int64_t u_hi, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > u_hi - u_lo) nthreads = (int)(u_hi - u_lo);
  if (nthreads < 1) return;
  layer_job jobs[512];
  pthread_t th[512];
  int live[512];
  for (int t = 0; t < nthreads; ++t) {
    layer_job J = {s, q_spec, q, K, V, idx, sel, lse, gap, out,
                   u_lo + (u_hi - u_lo) * t / nthreads, u_lo + (u_hi - u_lo) * (t + 1) / nthreads};
    jobs[t] = J;
    live[t] = (nthreads > 1) && pthread_create(&th[t], NULL, layer_worker, &jobs[t]) == 0;
    if (!live[t]) layer_worker(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (live[t]) pthread_join(th[t], NULL);
}

/* ---------------- landmark (chunk) selection ----------------
 *
 * The DualDecoder paper (Sec. 1) computes the retrieval index from the token
 * being processed and static GPU-resident KV landmarks; Sec. 2.2 describes
 * chunks of adjacent KV entries, each with a compressed landmark, the GPU
 * selecting chunks for the current query and retrieving their entries.  The
 * landmark itself is not specified; here it is the mean of the chunk's keys.
 * With chunk size c, the candidate positions [0, n - W) form M = (n - W) / c
 * chunks (c divides n - W and k):
 *   L_m   = (1/c) sum_{r < c} K[m c + r]                       (landmark)
 *   s_h,m = q_spec[h] . L_m / sqrt(d_k), alpha_h = softmax over m
 *   a_m   = alpha_m (MHA) or sum over the group of alpha_h,m
 *   the k / c chunks with the largest a_m (ties to the lower m) are selected,
 *   and the selected rows are every position of those chunks, ascending.
 */

/* Landmarks of unit (b, hk): L is [M][d]. */
void orc_landmarks_unit(const orc_shape* s, int chunk, const void* K, int b, int hk, double* L) {
  const int d = s->head_dim, n = s->ctx_len, M = (s->ctx_len - s->window) / chunk;
  const int64_t row0 = ((int64_t)b * s->n_kv_heads + hk) * n;
  for (int m = 0; m < M; ++m)
    for (int t = 0; t < d; ++t) {
      double acc = 0.0;
      for (int r = 0; r < chunk; ++r) acc += widen(K, s->dtype, (row0 + (int64_t)m * chunk + r) * d + t);
      L[(int64_t)m * d + t] = acc / chunk;
    }
}

/*
 * Chunk selection of unit (b, hk) from its landmarks L ([M][d]).  Writes the
 * k selected rows (ascending) to rows, the selected chunks' scores a_m to
 * sel ([k / c], ascending chunk order, may be NULL), the chunks' LSE per query
 * head of the group to lse ([G], may be NULL) and the relative gap between the
 * (k/c)-th and (k/c + 1)-th chunk score to *gap (may be NULL).
 */
void orc_landmark_select_unit(const orc_shape* s, int chunk, const void* q_spec, const double* L,
                              int b, int hk, int32_t* rows, double* sel, double* lse, double* gap) {
  const int G = group_size(s), d = s->head_dim, M = (s->ctx_len - s->window) / chunk;
  const int kc = s->top_k / chunk;
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  double* lg = (double*)malloc(sizeof(double) * (size_t)M);
  double* a = (double*)calloc((size_t)M, sizeof(double));
  for (int g = 0; g < G; ++g) {
    const int h = hk * G + g;
    const int64_t q_off = ((int64_t)b * s->n_q_heads + h) * d;
    double mx = -INFINITY;
    for (int m = 0; m < M; ++m) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += widen(q_spec, s->dtype, q_off + t) * L[(int64_t)m * d + t];
      lg[m] = acc * inv_sqrt_d;
      if (lg[m] > mx) mx = lg[m];
    }
    double sum = 0.0;
    for (int m = 0; m < M; ++m) sum += exp(lg[m] - mx);
    const double l = mx + log(sum);
    if (lse) lse[g] = l;
    for (int m = 0; m < M; ++m) a[m] += exp(lg[m] - l);
  }
  cand* c = (cand*)malloc(sizeof(cand) * (size_t)M);
  for (int m = 0; m < M; ++m) {
    c[m].a = a[m];
    c[m].j = m;
  }
  qsort(c, (size_t)M, sizeof(cand), by_score_desc);
  if (gap) *gap = (kc < M) ? (c[kc - 1].a - c[kc].a) / c[kc - 1].a : INFINITY;
  qsort(c, (size_t)kc, sizeof(cand), by_index_asc);
  for (int i = 0; i < kc; ++i) {
    if (sel) sel[i] = c[i].a;
    for (int r = 0; r < chunk; ++r) rows[i * chunk + r] = c[i].j * chunk + r;
  }
  free(c);
  free(a);
  free(lg);
}
