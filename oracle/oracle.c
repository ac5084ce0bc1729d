/*
 * Plain fp64 CPU oracle for mean-query column-sparse (Mx1-slice) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg load this library.  It shares no code,
 * header, table or constant with the CUDA path and is deliberately slow:
 * every quantity is the textbook definition evaluated in double precision,
 * one (batch, head, query group) unit at a time.
 *
 * What it follows (page titles as cited throughout this project):
 *  - "FG-Attn: Leveraging Fine-Grained Sparse Attention in Video Diffusion
 *    Models" (Pith review), sections "The pith" and referee comment 2 /
 *    §4.4: a group of M contiguous queries shares one key list (an Mx1
 *    slice per kept key); the list is chosen by scoring keys with the
 *    group's average query, k . q_avg / sqrt(D), against a threshold.
 *  - "Chipmunk: Training-Free Acceleration of Diffusion Transformers with
 *    Dynamic Column-Sparse Deltas" (Pith review), "What carries the
 *    argument" and major comment 1 (Alg. 3): [C,1] column sparsity with a
 *    top-k index mask; the deployed softmax is renormalised over the
 *    selected keys only (restricted softmax), not a masked full softmax.
 *  - LoSA abstract (mlsift.com diffusion-transformers list): keep the
 *    smallest key set whose attention mass reaches 99 %.
 *  - woonyee.org "DiT" page, section "Self Attention" / "Online Softmax":
 *    O = softmax(S) V with S = Q K^T / sqrt(d) per head; the oracle uses the
 *    plain two-pass form (row max, then sums) rather than the online update.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - scale s = 1/sqrt(d); LSE is the natural log of sum exp(s q.k) over the
 *    kept keys; an empty list gives o = 0 and lse = -inf.
 *  - group g covers query rows [g*M, min((g+1)*M, Nq)); the mean is over the
 *    rows that exist.
 *  - keys are ranked by (score descending, key index ascending).
 *  - THRESHOLD keeps j with p_j = exp(sigma_j - LSE_all) >= tau, where
 *    LSE_all is over all Nk keys; if none qualifies the top-ranked key is kept.
 *  - MASS keeps the shortest ranked prefix whose sum of p_j reaches rho
 *    (all keys if the total falls short through rounding, and all keys for
 *    rho >= 1, since every p_j is positive).
 *  - the reported cut is the score of the last key taken (TOPK, MASS) or
 *    ln(tau) + LSE_all (THRESHOLD).
 *  - dense-step lists (FG-Attn review, cached mask, "free parameters" and
 *    Fig. 10: keep a slice when at least one of its full-attention scores
 *    reaches tau_cached = 0.5/N; Chipmunk review, major comment 2 / Alg. 4:
 *    top-k columns by column sums of the attention probabilities, with the
 *    softmax constants of an earlier step): per group and key, the maximum
 *    (or the sum) over the group's queries of p_ij = exp(s q_i.k_j - lse_i),
 *    with lse_i supplied by the caller (the dense step's row log-sum-exp);
 *    rows whose lse is not finite contribute nothing.  The lists rank keys by
 *    ln of that statistic; LEVEL keeps keys whose statistic reaches tau.
 *  - sparse-delta attention (Chipmunk review, "What carries the argument",
 *    Eq. 1 as the referee reads it, and Appendix B.2: reuse the previous
 *    step's softmax normalisation): o_i = base_i + sign * sum over kept j of
 *    exp(s q_i.k_j - lse_i) v_j, with lse_i supplied; no renormalisation.
 *
 * Inputs are bf16 bit patterns (uint16) in [B, H, N, d] row-major order;
 * every bf16 value converts to double exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_TOPK 0
#define ORACLE_THRESHOLD 1
#define ORACLE_MASS 2
#define ORACLE_LEVEL 3
#define ORACLE_STAT_MAX 0
#define ORACLE_STAT_SUM 1

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------ threading */
typedef void (*unit_fn)(void* ctx, int64_t i);
typedef struct {
  unit_fn fn;
  void* ctx;
  int64_t begin, end;
} span_t;

static void* run_span(void* arg) {
  span_t* s = (span_t*)arg;
  for (int64_t i = s->begin; i < s->end; ++i) s->fn(s->ctx, i);
  return NULL;
}

/* Calls fn(ctx, i) for i in [0, n) on up to nthreads threads, contiguous
 * spans.  Each unit's arithmetic is independent of the split. */
static int parallel_for(int64_t n, int nthreads, unit_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  pthread_t tid[256];
  span_t spans[256];
  int created[256];
  for (int t = 0; t < nthreads; ++t) {
    spans[t].fn = fn;
    spans[t].ctx = ctx;
    spans[t].begin = n * t / nthreads;
    spans[t].end = n * (t + 1) / nthreads;
    created[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t)
    created[t] = pthread_create(&tid[t], NULL, run_span, &spans[t]) == 0;
  run_span(&spans[0]);
  for (int t = 1; t < nthreads; ++t)
    if (!created[t]) run_span(&spans[t]);
  for (int t = 1; t < nthreads; ++t)
    if (created[t]) pthread_join(tid[t], NULL);
  return 0;
}

/* ------------------------------------------------------------ geometry */
typedef struct {
  int64_t B, H, Nq, Nk, d, M;
} shape_t;

static int64_t num_groups(const shape_t* s) { return (s->Nq + s->M - 1) / s->M; }

/* unit u = (b*H + h)*G + g  ->  head offset (b*H + h) and group g */
static void split_unit(const shape_t* s, int64_t u, int64_t* bh, int64_t* g) {
  int64_t G = num_groups(s);
  *bh = u / G;
  *g = u % G;
}

/* ------------------------------------------------------------ mean query */
/* q_avg_g = (1/|g|) * sum_{i in g} q_i: the group's mean query (FG-Attn review, §4.4). */
static void mean_query_unit(const shape_t* s, const uint16_t* q, int64_t u, double* out) {
  int64_t bh, g;
  split_unit(s, u, &bh, &g);
  int64_t r0 = g * s->M;
  int64_t r1 = r0 + s->M < s->Nq ? r0 + s->M : s->Nq;
  for (int64_t c = 0; c < s->d; ++c) out[c] = 0.0;
  for (int64_t r = r0; r < r1; ++r) {
    const uint16_t* row = q + (bh * s->Nq + r) * s->d;
    for (int64_t c = 0; c < s->d; ++c) out[c] += bf16_value(row[c]);
  }
  double n = (double)(r1 - r0);
  for (int64_t c = 0; c < s->d; ++c) out[c] /= n;
}

typedef struct {
  shape_t s;
  const uint16_t *q, *k;
  double scale;
  const int64_t* units;
  double* out;
} score_ctx;

static void score_unit(void* vctx, int64_t i) {
  score_ctx* c = (score_ctx*)vctx;
  const shape_t* s = &c->s;
  int64_t u = c->units[i];
  int64_t bh, g;
  split_unit(s, u, &bh, &g);
  double* qbar = (double*)malloc(sizeof(double) * (size_t)s->d);
  mean_query_unit(s, c->q, u, qbar);
  double* dst = c->out + i * s->Nk;
  for (int64_t j = 0; j < s->Nk; ++j) {
    const uint16_t* krow = c->k + (bh * s->Nk + j) * s->d;
    double dot = 0.0;
    for (int64_t e = 0; e < s->d; ++e) dot += qbar[e] * bf16_value(krow[e]);
    dst[j] = c->scale * dot;  /* sigma_j = s * (q_avg . k_j) */
  }
  free(qbar);
}

/* Mean query of each listed unit: out[i*d + c]. */
int oracle_mean_query(const uint16_t* q, int64_t B, int64_t H, int64_t Nq, int64_t d,
                      int64_t M, const int64_t* units, int64_t n_units, double* out) {
  shape_t s = {B, H, Nq, 0, d, M};
  if (!q || !units || !out || M <= 0 || d <= 0) return 1;
  for (int64_t i = 0; i < n_units; ++i) mean_query_unit(&s, q, units[i], out + i * d);
  return 0;
}

/* Mean-query scores of each listed unit against all Nk keys:
 * out[i*Nk + j] = scale * (q_avg(unit i) . k_j). */
int oracle_group_scores(const uint16_t* q, const uint16_t* k, int64_t B, int64_t H,
                        int64_t Nq, int64_t Nk, int64_t d, int64_t M, double scale,
                        const int64_t* units, int64_t n_units, double* out, int nthreads) {
  if (!q || !k || !units || !out || M <= 0 || d <= 0 || Nk < 0) return 1;
  score_ctx c = {{B, H, Nq, Nk, d, M}, q, k, scale, units, out};
  return parallel_for(n_units, nthreads, score_unit, &c);
}

/* ------------------------------------------------------------ selection */
typedef struct {
  double score;
  int32_t index;
} ranked_t;

/* Rank order: score descending, then key index ascending. */
static int rank_cmp(const void* a, const void* b) {
  const ranked_t* x = (const ranked_t*)a;
  const ranked_t* y = (const ranked_t*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->index > y->index) - (x->index < y->index);
}

static int index_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct {
  const double* scores;
  int64_t Nk;
  int mode;
  int64_t topk;
  double tau, rho;
  int64_t* counts;
  int32_t* idx;
  double* cut;
} select_ctx;

static void select_row(void* vctx, int64_t r) {
  select_ctx* c = (select_ctx*)vctx;
  const int64_t Nk = c->Nk;
  const double* sc = c->scores + r * Nk;
  int32_t* out = c->idx + r * Nk;
  if (Nk == 0) {
    c->counts[r] = 0;
    c->cut[r] = -INFINITY;
    return;
  }
  ranked_t* order = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)Nk);
  for (int64_t j = 0; j < Nk; ++j) {
    order[j].score = sc[j];
    order[j].index = (int32_t)j;
  }
  qsort(order, (size_t)Nk, sizeof(ranked_t), rank_cmp);

  int64_t n = 0;
  double cut = 0.0;
  if (c->mode == ORACLE_TOPK) {
    n = c->topk < Nk ? c->topk : Nk;
    if (n < 1) n = 1;
    cut = order[n - 1].score;
  } else if (c->mode == ORACLE_LEVEL) {
    /* the statistic exp(score) itself reaches tau; a prefix of the ranking */
    while (n < Nk && exp(order[n].score) >= c->tau) ++n;
    if (n < 1) n = 1;
    cut = log(c->tau);
  } else {
    /* LSE over all keys: max, then the sum of exp(sigma - max). */
    double m = order[0].score;
    double z = 0.0;
    for (int64_t j = 0; j < Nk; ++j) z += exp(sc[j] - m);
    double lse = m + log(z);
    if (c->mode == ORACLE_THRESHOLD) {
      /* p_j >= tau; p decreases along the ranked order, so this is a prefix. */
      while (n < Nk && exp(order[n].score - lse) >= c->tau) ++n;
      if (n < 1) n = 1;
      cut = log(c->tau) + lse;
    } else {
      /* shortest ranked prefix with sum p >= rho; rho >= 1 needs every key,
       * since each p_j is positive */
      double acc = 0.0;
      if (c->rho >= 1.0) n = Nk;
      while (n < Nk) {
        acc += exp(order[n].score - lse);
        ++n;
        if (acc >= c->rho) break;
      }
      cut = order[n - 1].score;
    }
  }
  for (int64_t j = 0; j < n; ++j) out[j] = order[j].index;
  qsort(out, (size_t)n, sizeof(int32_t), index_cmp);
  c->counts[r] = n;
  c->cut[r] = cut;
  free(order);
}

/* Selects keys per row of scores[n_rows][Nk].  Kept indices, ascending, go to
 * idx[r*Nk ...]; counts[r] is their number; cut[r] the selection cut.
 * mode: 0 TOPK(topk), 1 THRESHOLD(tau), 2 MASS(rho), 3 LEVEL(tau): exp(score) >= tau. */
int oracle_select(const double* scores, int64_t n_rows, int64_t Nk, int mode, int64_t topk,
                  double tau, double rho, int64_t* counts, int32_t* idx, double* cut,
                  int nthreads) {
  if (!scores || !counts || !idx || !cut || mode < 0 || mode > 3) return 1;
  select_ctx c = {scores, Nk, mode, topk, tau, rho, counts, idx, cut};
  return parallel_for(n_rows, nthreads, select_row, &c);
}

/* ------------------------------------------------------------ attention */
typedef struct {
  shape_t s;
  const uint16_t *q, *k, *v;
  double scale;
  const int64_t* row_ptr;
  const int32_t* col_idx;
  const int64_t* units;
  double* o;
  double* lse;
} fwd_ctx;

/* Restricted softmax attention of one unit's queries over its kept keys:
 *   l_ij = s q_i.k_j,  m_i = max_j l_ij,  L_i = sum_j exp(l_ij - m_i),
 *   o_i = sum_j exp(l_ij - m_i) v_j / L_i,  lse_i = m_i + ln L_i. */
static void forward_unit(void* vctx, int64_t i) {
  fwd_ctx* c = (fwd_ctx*)vctx;
  const shape_t* s = &c->s;
  const int64_t d = s->d, M = s->M;
  int64_t u = c->units[i];
  int64_t bh, g;
  split_unit(s, u, &bh, &g);
  int64_t begin = c->row_ptr[u], end = c->row_ptr[u + 1];
  int64_t n = end > begin ? end - begin : 0;
  const int32_t* list = c->col_idx + begin;
  double* o_unit = c->o + i * M * d;
  double* lse_unit = c->lse + i * M;
  double* logits = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < M; ++r) {
    int64_t qi = g * M + r;
    double* orow = o_unit + r * d;
    for (int64_t e = 0; e < d; ++e) orow[e] = 0.0;
    if (qi >= s->Nq) {
      lse_unit[r] = 0.0;
      continue;
    }
    if (n == 0) {
      lse_unit[r] = -INFINITY;
      continue;
    }
    const uint16_t* qsrc = c->q + (bh * s->Nq + qi) * d;
    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      const uint16_t* krow = c->k + (bh * s->Nk + list[j]) * d;
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);
      logits[j] = c->scale * dot;
      if (logits[j] > m) m = logits[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      double p = exp(logits[j] - m);
      sum += p;
      const uint16_t* vrow = c->v + (bh * s->Nk + list[j]) * d;
      for (int64_t e = 0; e < d; ++e) orow[e] += p * bf16_value(vrow[e]);
    }
    for (int64_t e = 0; e < d; ++e) orow[e] /= sum;
    lse_unit[r] = m + log(sum);
  }
  free(qrow);
  free(logits);
}

/* Attention output of each listed unit: o[i][r][e] for r < M (rows past Nq
 * are zero), lse[i][r].  row_ptr has B*H*G+1 entries indexed by unit id. */
int oracle_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B,
                   int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t M, double scale,
                   const int64_t* row_ptr, const int32_t* col_idx, const int64_t* units,
                   int64_t n_units, double* o, double* lse, int nthreads) {
  if (!q || !k || !v || !row_ptr || !units || !o || !lse || M <= 0 || d <= 0) return 1;
  fwd_ctx c = {{B, H, Nq, Nk, d, M}, q, k, v, scale, row_ptr, col_idx, units, o, lse};
  return parallel_for(n_units, nthreads, forward_unit, &c);
}

/* ------------------------------------------------------------ dense-step statistics */
typedef struct {
  shape_t s;
  const uint16_t *q, *k;
  const double* lse;
  double scale;
  int stat;
  const int64_t* units;
  double* out;
} colstat_ctx;

/* For every key j: the maximum (stat 0) or the sum (stat 1) over the group's
 * query rows i of p_ij = exp(s q_i.k_j - lse_i); out holds its natural log. */
static void colstat_unit(void* vctx, int64_t i) {
  colstat_ctx* c = (colstat_ctx*)vctx;
  const shape_t* s = &c->s;
  const int64_t d = s->d;
  int64_t u = c->units[i];
  int64_t bh, g;
  split_unit(s, u, &bh, &g);
  int64_t r0 = g * s->M;
  int64_t r1 = r0 + s->M < s->Nq ? r0 + s->M : s->Nq;
  double* dst = c->out + i * s->Nk;
  double* qrows = (double*)malloc(sizeof(double) * (size_t)((r1 - r0) * d));
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t e = 0; e < d; ++e) qrows[(r - r0) * d + e] = bf16_value(c->q[(bh * s->Nq + r) * d + e]);
  for (int64_t j = 0; j < s->Nk; ++j) {
    const uint16_t* krow = c->k + (bh * s->Nk + j) * d;
    double stat = 0.0;
    for (int64_t r = r0; r < r1; ++r) {
      double lse = c->lse[bh * s->Nq + r];
      if (!isfinite(lse)) continue;
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += qrows[(r - r0) * d + e] * bf16_value(krow[e]);
      double p = exp(c->scale * dot - lse);
      if (c->stat == ORACLE_STAT_MAX) {
        if (p > stat) stat = p;
      } else {
        stat += p;
      }
    }
    dst[j] = log(stat);
  }
  free(qrows);
}

/* Column statistics of the listed units: out[i*Nk + j] = ln stat_j.
 * lse: double [B, H, Nq], natural-log row log-sum-exp of the dense step. */
int oracle_column_stats(const uint16_t* q, const uint16_t* k, const double* lse, int64_t B,
                        int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t M, double scale,
                        int stat, const int64_t* units, int64_t n_units, double* out,
                        int nthreads) {
  if (!q || !k || !lse || !units || !out || M <= 0 || d <= 0 || Nk < 0) return 1;
  if (stat != ORACLE_STAT_MAX && stat != ORACLE_STAT_SUM) return 1;
  colstat_ctx c = {{B, H, Nq, Nk, d, M}, q, k, lse, scale, stat, units, out};
  return parallel_for(n_units, nthreads, colstat_unit, &c);
}

/* ------------------------------------------------------------ sparse delta */
typedef struct {
  shape_t s;
  const uint16_t *q, *k, *v;
  double scale;
  const int64_t* row_ptr;
  const int32_t* col_idx;
  const double* lse;
  const double* base;
  double sign;
  const int64_t* units;
  double* o;
} delta_ctx;

/* o_i = base_i + sign * sum_{j in list} exp(s q_i.k_j - lse_i) v_j for the
 * rows of one unit (rows past Nq are zero; a row whose lse is not finite
 * keeps base_i). */
static void delta_unit(void* vctx, int64_t i) {
  delta_ctx* c = (delta_ctx*)vctx;
  const shape_t* s = &c->s;
  const int64_t d = s->d, M = s->M;
  int64_t u = c->units[i];
  int64_t bh, g;
  split_unit(s, u, &bh, &g);
  int64_t begin = c->row_ptr[u], end = c->row_ptr[u + 1];
  int64_t n = end > begin ? end - begin : 0;
  const int32_t* list = c->col_idx + begin;
  double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < M; ++r) {
    int64_t qi = g * M + r;
    double* orow = c->o + (i * M + r) * d;
    for (int64_t e = 0; e < d; ++e) orow[e] = 0.0;
    if (qi >= s->Nq) continue;
    if (c->base)
      for (int64_t e = 0; e < d; ++e) orow[e] = c->base[(bh * s->Nq + qi) * d + e];
    double lse = c->lse[bh * s->Nq + qi];
    if (!isfinite(lse)) continue;
    const uint16_t* qsrc = c->q + (bh * s->Nq + qi) * d;
    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);
    for (int64_t j = 0; j < n; ++j) {
      const uint16_t* krow = c->k + (bh * s->Nk + list[j]) * d;
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);
      double p = exp(c->scale * dot - lse);
      const uint16_t* vrow = c->v + (bh * s->Nk + list[j]) * d;
      for (int64_t e = 0; e < d; ++e) orow[e] += c->sign * p * bf16_value(vrow[e]);
    }
  }
  free(qrow);
}

/* Sparse-delta attention of the listed units: o[i][r][e] for r < M.
 * lse: double [B, H, Nq]; base: double [B, H, Nq, d] or NULL (zero). */
int oracle_forward_delta(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B,
                         int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t M, double scale,
                         const int64_t* row_ptr, const int32_t* col_idx, const double* lse,
                         const double* base, double sign, const int64_t* units, int64_t n_units,
                         double* o, int nthreads) {
  if (!q || !k || !v || !row_ptr || !col_idx || !lse || !units || !o || M <= 0 || d <= 0) return 1;
  delta_ctx c = {{B, H, Nq, Nk, d, M}, q, k, v, scale, row_ptr, col_idx, lse, base, sign, units, o};
  return parallel_for(n_units, nthreads, delta_unit, &c);
}
