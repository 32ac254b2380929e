/*
 * spec_verify_oracle.c -- plain, slow, scalar fp64 oracle.
 *
 * TEST INFRASTRUCTURE ONLY (see spec_verify_oracle.h).  Rows are independent;
 * the only parallelism is that whole rows are handed to POSIX threads, each
 * row computed by exactly the same scalar code.
 *
 * Sources (page title, section):
 *  [UNO]  "Uno: the draft model was already inside the target model",
 *         section "What 'lossless' actually has to mean": accept with
 *         probability min(1, p/q); on rejection resample from max(p - q, 0)
 *         renormalised; Uno's _sparse_verify_tensors fragment (gather by id
 *         equality, ratio = p/q if q > 0 else 0, accept iff u < min(1, ratio),
 *         correction probs = clamp(clean_probs - q_on_clean, 0) renormalised).
 *  [DF4]  DFlash/DFlash2 speculative decoding guide, 4.4 "Mathematical
 *         Losslessness Guarantee": target scores all positions in parallel;
 *         on a rejection at k the sequence is truncated at k and a replacement
 *         is drawn from the normalised residual.
 *  [DF2]  same guide, section 2 "Speculative Decoding Speedup Formulation":
 *         tau in [1, gamma + 1] including the target's bonus token.
 *  [DF4g] same guide, 4.4: under greedy decoding (T = 0) a draft token is
 *         accepted if and only if a condition holds whose formula did not
 *         survive on the page (see oracle_verify_greedy for the reading).
 *  [SDAR] "SDAR" page, section 5 (decoding timeline): each pass gives a full
 *         distribution at every masked position of the block; positions
 *         whose confidence clears a threshold tau are committed, at least
 *         the most confident one, so progress is guaranteed.
 *  [TKP]  Uno article (the test setting: temperature 1, top-k 50, top-p
 *         0.95) and DFlash/DFlash2 guide, Q3 (temperature scaling of both
 *         logit sets before the acceptance ratio; the formula is lost).
 *  [SSMD] "Self-Speculative Masked Diffusions", key design 2: verification
 *         in sigma order from the first unknown position; at the first
 *         rejection resample from max(0, target - draft) and end the round.
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *  - the accept comparison is strict, u < min(1, ratio) (Uno's `lt`);
 *  - one sample uniform per row, used only at the stop position;
 *  - inverse CDF in ascending vocabulary id (sparse: list order, which is
 *    ascending id): the token is the smallest y whose inclusive prefix sum
 *    exceeds u * T; if rounding leaves no such y, the last y with r(y) > 0;
 *  - residual mass T <= 0 after a rejection (impossible in exact arithmetic):
 *    draw from p of that position instead and flag the row;
 *  - -inf logits are allowed (probability 0); a NaN logit, a +inf logit or a
 *    row whose logits are all -inf is an input error for the whole row.
 */
#include "spec_verify_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* Exact widening: bf16 bits -> fp32 by a 16-bit shift -> double.       */
/* ------------------------------------------------------------------ */
static double widen(const void* base, int dtype, size_t i) {
  float f;
  if (dtype == ORACLE_BF16) {
    uint32_t w = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    memcpy(&f, &w, sizeof f);
  } else {
    f = ((const float*)base)[i];
  }
  return (double)f;
}

/* A logit row is usable if it has no NaN, no +inf and at least one finite
 * entry.  Returns 0 if usable, -1 otherwise. */
static int check_row(const void* base, int dtype, size_t off, int V) {
  int finite = 0;
  for (int y = 0; y < V; ++y) {
    double v = widen(base, dtype, off + (size_t)y);
    if (isnan(v) || v == INFINITY) return -1;
    if (v != -INFINITY) finite = 1;
  }
  return finite ? 0 : -1;
}

/* p = softmax(row), two-pass max-subtracted, in double. */
static void softmax_row(const void* base, int dtype, size_t off, int V, double* p) {
  double m = -INFINITY;
  for (int y = 0; y < V; ++y) {
    double v = widen(base, dtype, off + (size_t)y);
    if (v > m) m = v;
  }
  double s = 0.0;
  for (int y = 0; y < V; ++y) {
    p[y] = exp(widen(base, dtype, off + (size_t)y) - m);
    s += p[y];
  }
  for (int y = 0; y < V; ++y) p[y] /= s;
}

/* Accept test [UNO]: ratio = p/q if q > 0 else 0; accept iff u < min(1, ratio). */
static int accept_test(double px, double qx, float u, double* a_out, uint32_t* flag) {
  double ratio = (qx > 0.0) ? px / qx : 0.0;
  double a = ratio < 1.0 ? ratio : 1.0;
  double ud = (double)u;
  if (fabs(ud - a) < ORACLE_ACCEPT_BAND) *flag |= ORACLE_FLAG_ACCEPT_BAND;
  if (a_out) *a_out = a;
  return ud < a;
}

/* Inverse CDF over non-negative weights w[0..n) with uniform u.
 * T = sequential sum; the token is the smallest y with C(y) > u*T.
 * Returns the index, or -1 if T <= 0 (caller decides the fallback). */
static int inverse_cdf(const double* w, int n, float u, double* T_out, uint32_t* flag) {
  double T = 0.0;
  for (int y = 0; y < n; ++y) T += w[y];
  if (T_out) *T_out = T;
  if (!(T > 0.0)) return -1;
  double target = (double)u * T;
  double C = 0.0, Cprev = 0.0;
  int last_pos = -1;
  for (int y = 0; y < n; ++y) {
    if (w[y] > 0.0) last_pos = y;
    Cprev = C;
    C += w[y];
    if (C > target) {
      if (target - Cprev < ORACLE_TIE_BAND * T || C - target < ORACLE_TIE_BAND * T)
        *flag |= ORACLE_FLAG_CDF_TIE;
      return y;
    }
  }
  /* u*T >= final prefix: only through rounding. Clamp and flag. */
  *flag |= ORACLE_FLAG_CDF_TIE;
  return last_pos;
}

/* ------------------------------------------------------------------ */
/* Row-parallel driver                                                   */
/* ------------------------------------------------------------------ */
typedef void (*row_fn)(const void* args, int b, double* scratch);

typedef struct {
  row_fn fn;
  const void* args;
  int b0, b1;
  size_t scratch_doubles;
  int failed;
} worker_t;

static void* worker_main(void* p) {
  worker_t* w = (worker_t*)p;
  double* scratch = (double*)malloc(w->scratch_doubles * sizeof(double));
  if (!scratch) {
    w->failed = 1;
    return NULL;
  }
  for (int b = w->b0; b < w->b1; ++b) w->fn(w->args, b, scratch);
  free(scratch);
  return NULL;
}

int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static int run_rows(row_fn fn, const void* args, int B, size_t scratch_doubles, int nthreads) {
  if (B <= 0) return 0;
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if (nthreads > B) nthreads = B;
  worker_t* ws = (worker_t*)calloc((size_t)nthreads, sizeof(worker_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!ws || !th) {
    free(ws);
    free(th);
    return -1;
  }
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    ws[t].fn = fn;
    ws[t].args = args;
    ws[t].b0 = (int)((long long)B * t / nthreads);
    ws[t].b1 = (int)((long long)B * (t + 1) / nthreads);
    ws[t].scratch_doubles = scratch_doubles;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t, ++started)
    if (pthread_create(&th[t], NULL, worker_main, &ws[t]) != 0) break;
  worker_main(&ws[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  if (started != nthreads - 1) {
    /* thread creation failed: finish the remaining ranges here */
    for (int t = started + 1; t < nthreads; ++t) worker_main(&ws[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (ws[t].failed) rc = -1;
  free(ws);
  free(th);
  return rc;
}

/* ------------------------------------------------------------------ */
/* Dense                                                                 */
/* ------------------------------------------------------------------ */
typedef struct {
  const void *lt, *ld;
  int dtype;
  const int32_t* x;
  const float *u_acc, *u_s;
  int B, G, V;
  int32_t *n_out, *tok_out;
  double *resid_out, *acc_out, *T_out;
  uint32_t* flags;
} dense_args;

static void dense_row(const void* pa, int b, double* scratch) {
  const dense_args* a = (const dense_args*)pa;
  const int G = a->G, V = a->V;
  double* p = scratch;     /* [V] */
  double* q = scratch + V; /* [V] */
  double* w = q + V;       /* [V] */
  uint32_t flag = 0;
  const size_t trow = (size_t)b * (size_t)(G + 1);
  const size_t drow = (size_t)b * (size_t)G;
  int32_t* tok = a->tok_out + (size_t)b * (size_t)(G + 1);

  /* Input validation covers every row the parallel step reads. */
  int bad = 0;
  for (int j = 0; j <= G && !bad; ++j)
    bad |= check_row(a->lt, a->dtype, (trow + j) * (size_t)V, V);
  for (int j = 0; j < G && !bad; ++j) {
    bad |= check_row(a->ld, a->dtype, (drow + j) * (size_t)V, V);
    int32_t xj = a->x[drow + j];
    if (xj < 0 || xj >= V) bad = -1;
  }
  if (bad) {
    a->n_out[b] = -1;
    for (int j = 0; j <= G; ++j) tok[j] = -1;
    if (a->resid_out) memset(a->resid_out + (size_t)b * V, 0, sizeof(double) * (size_t)V);
    if (a->acc_out)
      for (int j = 0; j < G; ++j) a->acc_out[drow + j] = NAN;
    if (a->T_out) a->T_out[b] = NAN;
    if (a->flags) a->flags[b] = ORACLE_FLAG_INPUT_ERR;
    return;
  }

  /* Accept tests at every position (the target scored them all in
   * parallel [DF4]); the block stops at the first rejection. */
  int n = G;
  for (int j = 0; j < G; ++j) {
    softmax_row(a->lt, a->dtype, (trow + j) * (size_t)V, V, p);
    softmax_row(a->ld, a->dtype, (drow + j) * (size_t)V, V, q);
    int32_t xj = a->x[drow + j];
    double acc_p;
    uint32_t fj = 0;
    int acc = accept_test(p[xj], q[xj], a->u_acc[drow + j], &acc_p, &fj);
    if (a->acc_out) a->acc_out[drow + j] = acc_p;
    if (j <= n) flag |= fj; /* only decisions the sequential rule consumes */
    if (!acc && n == G) n = j;
  }

  int y;
  double T;
  if (n < G) {
    /* Residual at the first rejected position [UNO]. */
    softmax_row(a->lt, a->dtype, (trow + n) * (size_t)V, V, p);
    softmax_row(a->ld, a->dtype, (drow + n) * (size_t)V, V, q);
    for (int v = 0; v < V; ++v) {
      double r = p[v] - q[v];
      w[v] = r > 0.0 ? r : 0.0;
    }
    y = inverse_cdf(w, V, a->u_s[b], &T, &flag);
    if (y < 0) {
      flag |= ORACLE_FLAG_ZERO_RESID;
      memcpy(w, p, sizeof(double) * (size_t)V);
      y = inverse_cdf(w, V, a->u_s[b], &T, &flag);
    }
  } else {
    /* Bonus token from the target's distribution at position gamma [DF2]. */
    softmax_row(a->lt, a->dtype, (trow + G) * (size_t)V, V, w);
    y = inverse_cdf(w, V, a->u_s[b], &T, &flag);
  }

  a->n_out[b] = n;
  for (int j = 0; j < n; ++j) tok[j] = a->x[drow + j];
  tok[n] = y;
  for (int j = n + 1; j <= G; ++j) tok[j] = -1;
  if (a->resid_out) {
    double* ro = a->resid_out + (size_t)b * V;
    for (int v = 0; v < V; ++v) ro[v] = w[v] / T;
  }
  if (a->T_out) a->T_out[b] = T;
  if (a->flags) a->flags[b] = flag;
}

int oracle_verify_dense(const void* target_logits, const void* draft_logits, int dtype,
                        const int32_t* draft_ids, const float* u_accept, const float* u_sample,
                        int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                        double* residual_out, double* accept_prob, double* resid_mass,
                        uint32_t* flags, int nthreads) {
  if (B < 0 || gamma < 0 || V <= 0) return -1;
  if (B == 0) return 0;
  if (!target_logits || !u_sample || !n_accepted || !out_tokens) return -1;
  if (gamma > 0 && (!draft_logits || !draft_ids || !u_accept)) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  dense_args a = {target_logits, draft_logits, dtype,       draft_ids,  u_accept,
                  u_sample,      B,            gamma,       V,          n_accepted,
                  out_tokens,    residual_out, accept_prob, resid_mass, flags};
  return run_rows(dense_row, &a, B, 3 * (size_t)V, nthreads);
}

/* ------------------------------------------------------------------ */
/* Sparse top-k                                                          */
/* ------------------------------------------------------------------ */
typedef struct {
  const int32_t* tid;
  const float* tp;
  int kt;
  const int32_t* did;
  const float* dp;
  int kd;
  const int32_t* x;
  const float *u_acc, *u_s;
  int B, G, V;
  int32_t *n_out, *tok_out;
  double *resid_out, *acc_out, *T_out;
  uint32_t* flags;
} sparse_args;

static int check_list(const int32_t* ids, const float* pr, int k, int V) {
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0 || ids[i] >= V) return -1;
    if (i > 0 && ids[i] <= ids[i - 1]) return -1;
    if (!(pr[i] >= 0.0f) || isinf(pr[i])) return -1; /* NaN, negative or inf */
  }
  return 0;
}

/* Uno's gather: sum of the listed probabilities whose id equals x. */
static double gather_by_id(const int32_t* ids, const float* pr, int k, int32_t x) {
  double s = 0.0;
  for (int i = 0; i < k; ++i)
    if (ids[i] == x) s += (double)pr[i];
  return s;
}

static void sparse_row(const void* pa, int b, double* scratch) {
  const sparse_args* a = (const sparse_args*)pa;
  const int G = a->G, kt = a->kt, kd = a->kd;
  double* w = scratch; /* [kt] */
  uint32_t flag = 0;
  const size_t trow = (size_t)b * (size_t)(G + 1);
  const size_t drow = (size_t)b * (size_t)G;
  int32_t* tok = a->tok_out + (size_t)b * (size_t)(G + 1);

  int bad = 0;
  for (int j = 0; j <= G && !bad; ++j)
    bad |= check_list(a->tid + (trow + j) * kt, a->tp + (trow + j) * kt, kt, a->V);
  for (int j = 0; j < G && !bad; ++j) {
    bad |= check_list(a->did + (drow + j) * kd, a->dp + (drow + j) * kd, kd, a->V);
    if (a->x[drow + j] < 0 || a->x[drow + j] >= a->V) bad = -1;
  }
  if (bad) {
    a->n_out[b] = -1;
    for (int j = 0; j <= G; ++j) tok[j] = -1;
    if (a->resid_out) memset(a->resid_out + (size_t)b * kt, 0, sizeof(double) * (size_t)kt);
    if (a->acc_out)
      for (int j = 0; j < G; ++j) a->acc_out[drow + j] = NAN;
    if (a->T_out) a->T_out[b] = NAN;
    if (a->flags) a->flags[b] = ORACLE_FLAG_INPUT_ERR;
    return;
  }

  int n = G;
  for (int j = 0; j < G; ++j) {
    int32_t xj = a->x[drow + j];
    double p_spec = gather_by_id(a->tid + (trow + j) * kt, a->tp + (trow + j) * kt, kt, xj);
    double q_spec = gather_by_id(a->did + (drow + j) * kd, a->dp + (drow + j) * kd, kd, xj);
    double acc_p;
    uint32_t fj = 0;
    int acc = accept_test(p_spec, q_spec, a->u_acc[drow + j], &acc_p, &fj);
    if (a->acc_out) a->acc_out[drow + j] = acc_p;
    if (j <= n) flag |= fj;
    if (!acc && n == G) n = j;
  }

  const int32_t* tids = a->tid + (trow + n) * kt;
  const float* tps = a->tp + (trow + n) * kt;
  int yi;
  double T;
  if (n < G) {
    /* correction = clamp(clean_probs - q_on_clean, 0) on the target support */
    const int32_t* dids = a->did + (drow + n) * kd;
    const float* dps = a->dp + (drow + n) * kd;
    for (int i = 0; i < kt; ++i) {
      double q_on_clean = gather_by_id(dids, dps, kd, tids[i]);
      double r = (double)tps[i] - q_on_clean;
      w[i] = r > 0.0 ? r : 0.0;
    }
    yi = inverse_cdf(w, kt, a->u_s[b], &T, &flag);
    if (yi < 0) {
      flag |= ORACLE_FLAG_ZERO_RESID;
      for (int i = 0; i < kt; ++i) w[i] = (double)tps[i];
      yi = inverse_cdf(w, kt, a->u_s[b], &T, &flag);
    }
  } else {
    for (int i = 0; i < kt; ++i) w[i] = (double)tps[i];
    yi = inverse_cdf(w, kt, a->u_s[b], &T, &flag);
  }

  a->n_out[b] = n;
  for (int j = 0; j < n; ++j) tok[j] = a->x[drow + j];
  tok[n] = (yi >= 0) ? tids[yi] : -1;
  for (int j = n + 1; j <= G; ++j) tok[j] = -1;
  if (a->resid_out) {
    double* ro = a->resid_out + (size_t)b * kt;
    for (int i = 0; i < kt; ++i) ro[i] = (T > 0.0) ? w[i] / T : 0.0;
  }
  if (a->T_out) a->T_out[b] = T;
  if (yi < 0) flag |= ORACLE_FLAG_ZERO_RESID; /* all-zero target list */
  if (a->flags) a->flags[b] = flag;
}

int oracle_verify_sparse(const int32_t* tgt_ids, const float* tgt_probs, int kt,
                         const int32_t* drf_ids, const float* drf_probs, int kd,
                         const int32_t* draft_tokens, const float* u_accept, const float* u_sample,
                         int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                         double* residual_out, double* accept_prob, double* resid_mass,
                         uint32_t* flags, int nthreads) {
  if (B < 0 || gamma < 0 || V <= 0 || kt <= 0 || kd <= 0) return -1;
  if (B == 0) return 0;
  if (!tgt_ids || !tgt_probs || !u_sample || !n_accepted || !out_tokens) return -1;
  if (gamma > 0 && (!drf_ids || !drf_probs || !draft_tokens || !u_accept)) return -1;
  sparse_args a = {tgt_ids,  tgt_probs,  kt,        drf_ids,    drf_probs,
                   kd,       draft_tokens, u_accept, u_sample,  B,
                   gamma,    V,          n_accepted, out_tokens, residual_out,
                   accept_prob, resid_mass, flags};
  return run_rows(sparse_row, &a, B, (size_t)kt, nthreads);
}

/* ------------------------------------------------------------------ */
/* Any-order                                                             */
/* ------------------------------------------------------------------ */
typedef struct {
  const void *lt, *ld;
  int dtype;
  const int32_t *order, *tok_in;
  const float *u_acc, *u_s;
  int B, D, W, V;
  int32_t *n_out, *tok_out;
  double *resid_out, *acc_out, *T_out;
  uint32_t* flags;
} anyorder_args;

static void anyorder_row(const void* pa, int b, double* scratch) {
  const anyorder_args* a = (const anyorder_args*)pa;
  const int D = a->D, W = a->W, V = a->V;
  double* p = scratch;
  double* q = scratch + V;
  double* w = q + V;
  uint32_t flag = 0;
  const int32_t* sig = a->order + (size_t)b * W;
  const size_t base = (size_t)b * (size_t)D; /* row index of position 0 */
  int32_t* out = a->tok_out + base;

  int bad = 0;
  for (int i = 0; i < W && !bad; ++i) {
    int32_t s = sig[i];
    if (s < 0 || s >= D) {
      bad = -1;
      break;
    }
    for (int k = 0; k < i; ++k)
      if (sig[k] == s) bad = -1;
    if (bad) break;
    int32_t xs = a->tok_in[base + s];
    if (xs < 0 || xs >= V) bad = -1;
    bad |= check_row(a->lt, a->dtype, (base + s) * (size_t)V, V);
    bad |= check_row(a->ld, a->dtype, (base + s) * (size_t)V, V);
  }
  if (bad) {
    a->n_out[b] = -1;
    for (int i = 0; i < W; ++i)
      if (sig[i] >= 0 && sig[i] < D) out[sig[i]] = -1;
    if (a->resid_out) memset(a->resid_out + (size_t)b * V, 0, sizeof(double) * (size_t)V);
    if (a->acc_out)
      for (int i = 0; i < W; ++i) a->acc_out[(size_t)b * W + i] = NAN;
    if (a->T_out) a->T_out[b] = NAN;
    if (a->flags) a->flags[b] = ORACLE_FLAG_INPUT_ERR;
    return;
  }

  /* Verify in sigma order; the round ends at the first rejection [SSMD]. */
  int n = W;
  for (int i = 0; i < W; ++i) {
    int32_t s = sig[i];
    softmax_row(a->lt, a->dtype, (base + s) * (size_t)V, V, p);
    softmax_row(a->ld, a->dtype, (base + s) * (size_t)V, V, q);
    int32_t xs = a->tok_in[base + s];
    double acc_p;
    uint32_t fi = 0;
    int acc = accept_test(p[xs], q[xs], a->u_acc[(size_t)b * W + i], &acc_p, &fi);
    if (a->acc_out) a->acc_out[(size_t)b * W + i] = acc_p;
    if (i <= n) flag |= fi;
    if (!acc && n == W) n = i;
  }

  double T = 0.0;
  int y = -1;
  if (n < W) {
    int32_t s = sig[n];
    softmax_row(a->lt, a->dtype, (base + s) * (size_t)V, V, p);
    softmax_row(a->ld, a->dtype, (base + s) * (size_t)V, V, q);
    for (int v = 0; v < V; ++v) {
      double r = p[v] - q[v];
      w[v] = r > 0.0 ? r : 0.0;
    }
    y = inverse_cdf(w, V, a->u_s[b], &T, &flag);
    if (y < 0) {
      flag |= ORACLE_FLAG_ZERO_RESID;
      memcpy(w, p, sizeof(double) * (size_t)V);
      y = inverse_cdf(w, V, a->u_s[b], &T, &flag);
    }
  }

  a->n_out[b] = n;
  for (int i = 0; i < W; ++i) {
    int32_t s = sig[i];
    out[s] = (i < n) ? a->tok_in[base + s] : (i == n ? y : -1);
  }
  if (a->resid_out) {
    double* ro = a->resid_out + (size_t)b * V;
    for (int v = 0; v < V; ++v) ro[v] = (n < W) ? w[v] / T : 0.0;
  }
  if (a->T_out) a->T_out[b] = (n < W) ? T : 0.0;
  if (a->flags) a->flags[b] = flag;
}

int oracle_verify_anyorder(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* order, const int32_t* draft_tokens,
                           const float* u_accept, const float* u_sample, int B, int D, int W,
                           int V, int32_t* n_accepted, int32_t* out_tokens, double* residual_out,
                           double* accept_prob, double* resid_mass, uint32_t* flags,
                           int nthreads) {
  if (B < 0 || D <= 0 || W <= 0 || W > D || V <= 0) return -1;
  if (B == 0) return 0;
  if (!target_logits || !draft_logits || !order || !draft_tokens || !u_accept || !u_sample ||
      !n_accepted || !out_tokens)
    return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  anyorder_args a = {target_logits, draft_logits, dtype,      order,      draft_tokens,
                     u_accept,      u_sample,     B,          D,          W,
                     V,             n_accepted,   out_tokens, residual_out, accept_prob,
                     resid_mass,    flags};
  return run_rows(anyorder_row, &a, B, 3 * (size_t)V, nthreads);
}

/* ------------------------------------------------------------------ */
/* Greedy (T = 0)                                                        */
/* ------------------------------------------------------------------ */
/* [DF4g] Reading: the limit T -> 0 of the stochastic rule.  As T -> 0,
 * p_k = softmax(target[k] / T) becomes the point mass at a_k = argmax_y
 * target[k, y] (the smallest such y when several ids share the maximum), so
 *  - x_k is accepted iff x_k = a_k (then p_k(x_k) = 1 >= q_k(x_k); otherwise
 *    p_k(x_k) = 0 and the ratio is 0);
 *  - the block stops at the first k with x_k != a_k, and the replacement,
 *    drawn from max(p_k - q_k, 0) normalised, is the point mass at a_k;
 *  - if every draft is accepted the bonus is a_gamma.
 * No uniform is consumed.  Input errors as in the dense rule (NaN, +inf or
 * an all -inf target row, a draft id out of range). */
typedef struct {
  const void* lt;
  int dtype;
  const int32_t* x;
  int B, G, V;
  int32_t *n_out, *tok_out;
} greedy_args;

static int argmax_row(const void* base, int dtype, size_t off, int V) {
  int best = 0;
  double bv = widen(base, dtype, off);
  for (int y = 1; y < V; ++y) {
    double v = widen(base, dtype, off + (size_t)y);
    if (v > bv) {
      bv = v;
      best = y;
    }
  }
  return best;
}

static void greedy_row(const void* pa, int b, double* scratch) {
  const greedy_args* a = (const greedy_args*)pa;
  const int G = a->G, V = a->V;
  (void)scratch;
  const size_t trow = (size_t)b * (size_t)(G + 1);
  const size_t drow = (size_t)b * (size_t)G;
  int32_t* tok = a->tok_out + (size_t)b * (size_t)(G + 1);
  int bad = 0;
  for (int j = 0; j <= G && !bad; ++j)
    bad |= check_row(a->lt, a->dtype, (trow + j) * (size_t)V, V);
  for (int j = 0; j < G && !bad; ++j) {
    int32_t xj = a->x[drow + j];
    if (xj < 0 || xj >= V) bad = -1;
  }
  if (bad) {
    a->n_out[b] = -1;
    for (int j = 0; j <= G; ++j) tok[j] = -1;
    return;
  }
  int n = G;
  for (int j = 0; j < G; ++j)
    if (a->x[drow + j] != argmax_row(a->lt, a->dtype, (trow + j) * (size_t)V, V)) {
      n = j;
      break;
    }
  a->n_out[b] = n;
  for (int j = 0; j < n; ++j) tok[j] = a->x[drow + j];
  tok[n] = argmax_row(a->lt, a->dtype, (trow + n) * (size_t)V, V);
  for (int j = n + 1; j <= G; ++j) tok[j] = -1;
}

int oracle_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_ids, int B,
                         int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                         int nthreads) {
  if (B < 0 || gamma < 0 || V <= 0) return -1;
  if (B == 0) return 0;
  if (!target_logits || !n_accepted || !out_tokens) return -1;
  if (gamma > 0 && !draft_ids) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  greedy_args a = {target_logits, dtype, draft_ids, B, gamma, V, n_accepted, out_tokens};
  return run_rows(greedy_row, &a, B, 1, nthreads);
}

/* ------------------------------------------------------------------ */
/* Confidence-threshold commit [SDAR]                                   */
/* ------------------------------------------------------------------ */
/* Readings (the page states the rule in prose only): the confidence of a
 * masked position is its largest probability, max_y p_i(y) = 1 / sum_y
 * exp(l_y - max l); its candidate token is the argmax (smallest id on ties);
 * "clears tau" is conf > tau; "at least the argmax is" committed means that
 * when no masked position clears tau, the one with the largest confidence
 * (the smallest index on ties) is committed. */
typedef struct {
  const void* lt;
  int dtype;
  const int32_t* masked;
  double tau;
  int B, W, V;
  int32_t *commit, *tokens;
  double* conf;
  uint32_t* flags;
} commit_args;

static void commit_row(const void* pa, int b, double* p) {
  const commit_args* a = (const commit_args*)pa;
  const int W = a->W, V = a->V;
  int32_t* cm = a->commit + (size_t)b * W;
  int32_t* tk = a->tokens + (size_t)b * W;
  double* cf = a->conf ? a->conf + (size_t)b * W : NULL;
  uint32_t flag = 0;
  int bad = 0;
  for (int i = 0; i < W && !bad; ++i)
    if (a->masked[(size_t)b * W + i])
      bad |= check_row(a->lt, a->dtype, ((size_t)b * W + i) * (size_t)V, V);
  if (bad) {
    for (int i = 0; i < W; ++i) {
      cm[i] = -1;
      tk[i] = -1;
      if (cf) cf[i] = NAN;
    }
    if (a->flags) a->flags[b] = ORACLE_FLAG_INPUT_ERR;
    return;
  }
  int ncommit = 0, best = -1;
  double best_c = -1.0, second_c = -1.0;
  for (int i = 0; i < W; ++i) {
    cm[i] = 0;
    tk[i] = -1;
    if (cf) cf[i] = NAN;
    if (!a->masked[(size_t)b * W + i]) continue;
    const size_t off = ((size_t)b * W + i) * (size_t)V;
    softmax_row(a->lt, a->dtype, off, V, p);
    int y = 0;
    for (int v = 1; v < V; ++v)
      if (p[v] > p[y]) y = v;
    const double c = p[y];
    if (cf) cf[i] = c;
    if (fabs(c - a->tau) < ORACLE_ACCEPT_BAND) flag |= ORACLE_FLAG_ACCEPT_BAND;
    if (c > a->tau) {
      cm[i] = 1;
      tk[i] = y;
      ++ncommit;
    }
    if (c > best_c) {
      second_c = best_c;
      best_c = c;
      best = i;
    } else if (c > second_c) {
      second_c = c;
    }
  }
  if (ncommit == 0 && best >= 0) {  /* progress: the most confident position */
    const size_t off = ((size_t)b * W + best) * (size_t)V;
    softmax_row(a->lt, a->dtype, off, V, p);
    int y = 0;
    for (int v = 1; v < V; ++v)
      if (p[v] > p[y]) y = v;
    cm[best] = 1;
    tk[best] = y;
    if (second_c >= 0.0 && best_c - second_c <= ORACLE_TIE_BAND * best_c) flag |= ORACLE_FLAG_CDF_TIE;
  }
  if (a->flags) a->flags[b] = flag;
}

int oracle_commit_confident(const void* logits, int dtype, const int32_t* masked, double tau,
                            int B, int W, int V, int32_t* commit, int32_t* tokens,
                            double* confidence, uint32_t* flags, int nthreads) {
  if (B < 0 || W <= 0 || V <= 0) return -1;
  if (B == 0) return 0;
  if (!logits || !masked || !commit || !tokens) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  commit_args a = {logits, dtype, masked, tau, B, W, V, commit, tokens, confidence, flags};
  return run_rows(commit_row, &a, B, (size_t)V, nthreads);
}

/* ------------------------------------------------------------------ */
/* Sparse support from dense logits: temperature, top-k, top-p [TKP]    */
/* ------------------------------------------------------------------ */
/* Readings (the usual definitions, which the pages name but do not spell
 * out): the top-k set is the K largest logits (ties: smaller id first; the
 * order is the same for every T > 0); its probabilities are softmax(l / T)
 * renormalised over the set; top-p keeps, in decreasing probability (ties:
 * smaller id first), the shortest prefix whose cumulative mass reaches top_p
 * -- at least one entry -- and renormalises it; the other entries of the
 * set keep their ids with probability 0, so every row is a K-entry list in
 * ascending id order (the form the sparse verification takes). */
typedef struct {
  double v;
  int32_t id;
} vid_t;

static int vid_desc(const void* a, const void* b) {
  const vid_t* x = (const vid_t*)a;
  const vid_t* y = (const vid_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

typedef struct {
  double p;
  int32_t id;
} pid_t_;

static int pid_by_id(const void* a, const void* b) {
  const pid_t_* x = (const pid_t_*)a;
  const pid_t_* y = (const pid_t_*)b;
  return (x->id > y->id) - (x->id < y->id);
}

typedef struct {
  const void* lt;
  int dtype;
  int N, V, K;
  double T, top_p;
  int32_t* ids;
  double* probs;
  uint32_t* flags;
} support_args;

static void support_row(const void* pa, int r, double* scratch) {
  const support_args* a = (const support_args*)pa;
  const int V = a->V, K = a->K;
  int32_t* oid = a->ids + (size_t)r * K;
  double* op = a->probs + (size_t)r * K;
  const size_t off = (size_t)r * (size_t)V;
  if (check_row(a->lt, a->dtype, off, V)) {
    for (int i = 0; i < K; ++i) {
      oid[i] = -1;
      op[i] = NAN;
    }
    if (a->flags) a->flags[r] = ORACLE_FLAG_INPUT_ERR;
    return;
  }
  vid_t* all = (vid_t*)scratch; /* scratch holds 2V doubles: room for V pairs */
  for (int y = 0; y < V; ++y) {
    all[y].v = widen(a->lt, a->dtype, off + (size_t)y);
    all[y].id = y;
  }
  qsort(all, (size_t)V, sizeof(vid_t), vid_desc); /* the top-k set is all[0..K) */
  /* softmax over the set, in decreasing order (already sorted by value) */
  const double m = all[0].v / a->T;
  double Z = 0.0;
  pid_t_* set = (pid_t_*)malloc(sizeof(pid_t_) * (size_t)K);
  if (!set) return;
  for (int i = 0; i < K; ++i) {
    set[i].p = (all[i].v == -INFINITY) ? 0.0 : exp(all[i].v / a->T - m);
    set[i].id = all[i].id;
    Z += set[i].p;
  }
  for (int i = 0; i < K; ++i) set[i].p /= Z;
  /* top-p: shortest prefix (decreasing probability, ties by id: the same
   * order) with cumulative mass >= top_p, at least one entry */
  double c = 0.0;
  int keep = K;
  uint32_t flag = 0;
  for (int i = 0; i < K && a->top_p < 1.0; ++i) { /* top_p >= 1 keeps the whole set */
    c += set[i].p;
    if (c >= a->top_p) {
      keep = i + 1;
      if (c - a->top_p < ORACLE_TIE_BAND) flag |= ORACLE_FLAG_CDF_TIE;
      break;
    }
    if (a->top_p - c < ORACLE_TIE_BAND) flag |= ORACLE_FLAG_CDF_TIE;
  }
  double Zk = 0.0;
  for (int i = 0; i < keep; ++i) Zk += set[i].p;
  for (int i = 0; i < K; ++i) set[i].p = (i < keep) ? set[i].p / Zk : 0.0;
  qsort(set, (size_t)K, sizeof(pid_t_), pid_by_id);
  for (int i = 0; i < K; ++i) {
    oid[i] = set[i].id;
    op[i] = set[i].p;
  }
  free(set);
  if (a->flags) a->flags[r] = flag;
}

int oracle_support_topk(const void* logits, int dtype, int N, int V, double T, int K,
                        double top_p, int32_t* ids, double* probs, uint32_t* flags,
                        int nthreads) {
  if (N < 0 || V <= 0 || K < 1 || K > V || !(T > 0.0)) return -1;
  if (N == 0) return 0;
  if (!logits || !ids || !probs) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  support_args a = {logits, dtype, N, V, K, T, top_p, ids, probs, flags};
  return run_rows(support_row, &a, N, 2 * (size_t)V, nthreads);
}

/* ------------------------------------------------------------------ */
/* Windowed multi-round any-order verification                          */
/* ------------------------------------------------------------------ */
/* [SSMD4] ("Self-Speculative Masked Diffusions", key design 4, windowed
 * multi-round verification).  One non-causal pass gives the draft
 * distributions of the window W(i); several causal verification rounds then
 * run on them.  Each round verifies the still-masked window positions in
 * sigma order against that round's target distributions with that round's
 * draft tokens (after a resample the later drafts change, and the causal
 * probabilities are recomputed); it ends at its first rejection, whose
 * position is resampled from max(p - q, 0) renormalised and revealed (the
 * any-order rule, key design 2); the next round starts after it.  A round
 * that accepts every remaining draft closes the window.  No bonus token.
 *
 * Input errors are raised where the rounds use an input: an out-of-range or
 * repeated sigma entry inside the window (checked first), a revealed count
 * outside [0, D], a window below 1, and -- as the rounds reach them -- a
 * draft token out of range or a logit row with NaN, +inf or no finite
 * entry. */
typedef struct {
  const void *lt, *ld;
  int dtype;
  const int32_t *order, *i0, *win, *tok_in;
  const float *u_acc, *u_s;
  int B, R, D, V;
  int32_t *tok_out, *n_out, *racc_out;
  uint32_t* flags;
} rounds_args;

static void rounds_row(const void* pa, int b, double* scratch) {
  const rounds_args* a = (const rounds_args*)pa;
  const int R = a->R, D = a->D, V = a->V;
  double* p = scratch;
  double* q = p + V;
  double* w = q + V;
  uint32_t flag = 0;
  const int32_t* sig = a->order + (size_t)b * D;
  int32_t* out = a->tok_out + (size_t)b * D;
  int32_t* racc = a->racc_out + (size_t)b * R;
  const int i0 = a->i0[b], W = a->win[b];
  for (int r = 0; r < R; ++r) racc[r] = -1;

  int bad = (i0 < 0 || i0 > D || W < 1);
  const int e = bad ? 0 : ((W > D - i0) ? D : i0 + W); /* the window is sigma[i0, e) */
  for (int k = i0; k < e && !bad; ++k) {
    if (sig[k] < 0 || sig[k] >= D) bad = 1;
    for (int k2 = i0; k2 < k && !bad; ++k2)
      if (sig[k2] == sig[k]) bad = 1;
  }

  int i = i0; /* sigma index of the first still-masked window position */
  for (int r = 0; r < R && !bad && i < e; ++r) {
    const size_t rr = ((size_t)b * R + r) * (size_t)D; /* round r's [D] slice */
    const size_t dd = (size_t)b * (size_t)D;
    int stop = e;
    for (int k = i; k < e; ++k) {
      const int32_t s = sig[k];
      const int32_t x = a->tok_in[rr + s];
      if (x < 0 || x >= V || check_row(a->lt, a->dtype, (rr + s) * (size_t)V, V) ||
          check_row(a->ld, a->dtype, (dd + s) * (size_t)V, V)) {
        bad = 1;
        break;
      }
      softmax_row(a->lt, a->dtype, (rr + s) * (size_t)V, V, p);
      softmax_row(a->ld, a->dtype, (dd + s) * (size_t)V, V, q);
      if (!accept_test(p[x], q[x], a->u_acc[rr + k], NULL, &flag)) {
        stop = k; /* p and q now hold this position's distributions */
        break;
      }
    }
    if (bad) break;
    for (int k = i; k < stop; ++k) out[sig[k]] = a->tok_in[rr + sig[k]];
    racc[r] = stop - i;
    if (stop < e) {
      for (int v = 0; v < V; ++v) {
        const double d = p[v] - q[v];
        w[v] = d > 0.0 ? d : 0.0;
      }
      const float us = a->u_s[(size_t)b * R + r];
      int y = inverse_cdf(w, V, us, NULL, &flag);
      if (y < 0) {
        flag |= ORACLE_FLAG_ZERO_RESID;
        y = inverse_cdf(p, V, us, NULL, &flag);
      }
      out[sig[stop]] = y;
      i = stop + 1;
    } else {
      i = e;
    }
  }

  if (bad) {
    for (int k = (i0 >= 0 ? i0 : 0); k < e; ++k)
      if (sig[k] >= 0 && sig[k] < D) out[sig[k]] = -1;
    for (int r = 0; r < R; ++r) racc[r] = -1;
    a->n_out[b] = -1;
    if (a->flags) a->flags[b] = ORACLE_FLAG_INPUT_ERR;
    return;
  }
  a->n_out[b] = i;
  if (a->flags) a->flags[b] = flag;
}

int oracle_anyorder_rounds(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* order, const int32_t* revealed, const int32_t* window,
                           const int32_t* draft_tokens, const float* u_accept,
                           const float* u_sample, int B, int R, int D, int V, int32_t* tokens,
                           int32_t* n_revealed, int32_t* round_accepts, uint32_t* flags,
                           int nthreads) {
  if (B < 0 || R <= 0 || D <= 0 || V <= 0) return -1;
  if (B == 0) return 0;
  if (!target_logits || !draft_logits || !order || !revealed || !window || !draft_tokens ||
      !u_accept || !u_sample || !tokens || !n_revealed || !round_accepts)
    return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  rounds_args a = {target_logits, draft_logits, dtype,    order,      revealed,
                   window,        draft_tokens, u_accept, u_sample,   B,
                   R,             D,            V,        tokens,     n_revealed,
                   round_accepts, flags};
  return run_rows(rounds_row, &a, B, 3 * (size_t)V, nthreads);
}

/* [SSMD4] The window W(i) of the outer step that starts with i of D tokens
 * revealed: the page has it grow with i, cosine-shaped, set by dtau.  Reading:
 * the positions a cosine-schedule masked-diffusion sampler reveals over the
 * next dtau of its time.  Its revealed fraction at time t in [0, 1] is
 * f(t) = 1 - cos(pi t / 2) (slow at first, faster later); t(i) solves
 * f(t) = i / D; W(i) = ceil(D f(min(1, t(i) + dtau)) - 1e-9) - i, at least 1,
 * at most D - i (the 1e-9 keeps a product that rounds just above an integer
 * from adding a position).  0 when i >= D. */
int oracle_cosine_window(int D, int i, double dtau) {
  if (D <= 0 || i < 0) return -1;
  if (i >= D) return 0;
  const double pi = 3.14159265358979323846;
  const double t = (2.0 / pi) * acos(1.0 - (double)i / (double)D);
  double t1 = t + (dtau > 0.0 ? dtau : 0.0);
  if (t1 > 1.0) t1 = 1.0;
  const double reach = (double)D * (1.0 - cos(0.5 * pi * t1));
  long long end = (long long)ceil(reach - 1e-9);
  if (end > D) end = D;
  long long wv = end - i;
  if (wv < 1) wv = 1;
  return (int)wv;
}
