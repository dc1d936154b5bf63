/*
 * tdt_oracle.c -- plain CPU oracle for the Token-and-Duration Transducer (TDT)
 * loss and its gradient, in float64.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The product library
 * never loads this file and shares no code, header or constant with it.
 *
 * What it computes (sources, by page and section):
 *  - "tdt-loss: add TDT loss kernel" (kernels-community PR #882), list
 *    "What's in it": a log-softmax over the vocabulary at every lattice node,
 *    alpha/beta passes over the lattice accumulated in float64, one set of
 *    gradients w.r.t. the token and the duration logits, fp32/fp16/bf16
 *    logits read directly (also as a slice logits[..., :V] of a wider
 *    tensor), and the reductions mean_volume, mean_batch, mean, sum, none.
 *  - "Add TDT loss kernel" (transformers PR #46048), review thread: sigma
 *    (the logit under-normalisation) is a loss parameter that may be != 0;
 *    commit list: "-100 label padding", "separate pad token and blank token".
 *  The pages print no recursion.  This file follows the published TDT
 *  lattice (Xu et al. 2023, "Efficient Sequence Transduction by Jointly
 *  Predicting Tokens and Durations") in its plainest form:
 *    node (t,u), 0 <= t < T_b, 0 <= u <= U_b; durations d_0..d_{D-1};
 *    blank arc  (t,u) -> (t+d_i, u)    for d_i > 0, weight lpB(t,u)+lpD_i(t,u)-sigma;
 *    label arc  (t,u) -> (t+d_i, u+1)  for every d_i (0 included), u < U_b,
 *               weight lpL(t,u)+lpD_i(t,u)-sigma, lpL = log-softmax of label y_{u+1};
 *    a path starts at (0,0) and ends with a blank arc from (t,U_b) landing
 *    exactly on frame T_b; label arcs land on frames < T_b.
 *  lpB, lpL: log-softmax over the V token logits z[0..V) (blank inside);
 *  lpD_i:    log-softmax over the D duration logits z[V..V+D).
 *  L_b = -log sum over paths of exp(sum of arc weights).
 *
 * Everything is written out literally: log-sum-exp of a list of terms, the
 * alpha recursion in (t,u) order, the beta recursion in reverse order,
 * arc posteriors gamma = exp(alpha(src) + w + beta(dst) - logL), and
 * dL/dz = c_b * (softmax * N - [k = blank] * sum gamma_blank
 *                            - [k = label] * sum gamma_label).
 * OpenMP runs only over independent utterances or independent nodes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int64_t i64;

enum { OR_OK = 0, OR_EINVAL = -1, OR_ENOMEM = -2 };
enum { OR_RED_NONE = 0, OR_RED_SUM = 1, OR_RED_MEAN = 2, OR_RED_MEAN_BATCH = 3,
       OR_RED_MEAN_VOLUME = 4 };

/* log(sum_i exp(x_i)); the empty sum (all -inf) is -inf. */
static double log_sum_exp(const double *x, int n) {
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (x[i] > m) m = x[i];
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += exp(x[i] - m);
  return m + log(s);
}

typedef struct {
  const void *logits;
  int logits_f64; /* 1: double elements, 0: float elements */
  i64 B, T, U1, VD, V, D;
  i64 s0, s1, s2, s3; /* element strides */
  const i64 *labels;
  i64 labels_stride; /* elements between utterances in labels */
  const i64 *logit_lens, *label_lens;
  const int *dur;
  int blank;
  double sigma;
} problem;

static double z_at(const problem *p, i64 b, i64 t, i64 u, i64 k) {
  i64 off = b * p->s0 + t * p->s1 + u * p->s2 + k * p->s3;
  if (p->logits_f64) return ((const double *)p->logits)[off];
  return (double)((const float *)p->logits)[off];
}

static i64 node_id(const problem *p, i64 b, i64 t, i64 u) {
  return (b * p->T + t) * p->U1 + u;
}

/* An utterance is usable when its lengths fit the tensor and every label
 * it uses is a token other than blank (the reading of "-100 label padding":
 * entries at index >= U_b are ignored). */
static int utterance_valid(const problem *p, i64 b) {
  i64 Tb = p->logit_lens[b], Ub = p->label_lens[b];
  if (Tb < 1 || Tb > p->T || Ub < 0 || Ub > p->U1 - 1) return 0;
  for (i64 u = 0; u < Ub; ++u) {
    i64 y = p->labels[b * p->labels_stride + u];
    if (y < 0 || y >= p->V || y == p->blank) return 0;
  }
  return 1;
}

typedef struct {
  double *lse_tok, *lp_blank, *lp_label, *lp_dur; /* lp_dur: [node][D] */
} tables;

/* Per-node log-softmaxes ("log-softmax over the vocabulary for each lattice
 * node"; the duration head is normalised on its own). */
static void build_tables(const problem *p, const int *valid, tables *tb) {
  i64 nodes = p->B * p->T * p->U1;
#pragma omp parallel
  {
    double *buf = (double *)malloc(sizeof(double) * (size_t)(p->V > p->D ? p->V : p->D));
#pragma omp for schedule(static)
    for (i64 n = 0; n < nodes; ++n) {
      i64 b = n / (p->T * p->U1), t = (n / p->U1) % p->T, u = n % p->U1;
      tb->lse_tok[n] = NAN;
      tb->lp_blank[n] = NAN;
      tb->lp_label[n] = NAN;
      for (i64 i = 0; i < p->D; ++i) tb->lp_dur[n * p->D + i] = NAN;
      if (!valid[b] || t >= p->logit_lens[b] || u > p->label_lens[b]) continue;
      for (i64 k = 0; k < p->V; ++k) buf[k] = z_at(p, b, t, u, k);
      double lse = log_sum_exp(buf, (int)p->V);
      tb->lse_tok[n] = lse;
      tb->lp_blank[n] = buf[p->blank] - lse;
      if (u < p->label_lens[b]) {
        i64 y = p->labels[b * p->labels_stride + u];
        tb->lp_label[n] = buf[y] - lse;
      }
      for (i64 i = 0; i < p->D; ++i) buf[i] = z_at(p, b, t, u, p->V + i);
      double lse_d = log_sum_exp(buf, (int)p->D);
      for (i64 i = 0; i < p->D; ++i) tb->lp_dur[n * p->D + i] = buf[i] - lse_d;
    }
    free(buf);
  }
}

static double w_blank(const problem *p, const tables *tb, i64 n, i64 i) {
  return tb->lp_blank[n] + tb->lp_dur[n * p->D + i] - p->sigma;
}
static double w_label(const problem *p, const tables *tb, i64 n, i64 i) {
  return tb->lp_label[n] + tb->lp_dur[n * p->D + i] - p->sigma;
}

/* Forward variables: alpha(t,u) = log of the summed weight of all partial
 * paths from (0,0) to (t,u).  Returns log-likelihood of the utterance. */
static double run_alpha(const problem *p, const tables *tb, i64 b, double *alpha) {
  i64 Tb = p->logit_lens[b], Ub = p->label_lens[b];
  double *terms = (double *)malloc(sizeof(double) * (size_t)(2 * p->D + 1));
  for (i64 t = 0; t < Tb; ++t) {
    for (i64 u = 0; u <= Ub; ++u) {
      i64 n = node_id(p, b, t, u);
      if (t == 0 && u == 0) { alpha[n] = 0.0; continue; }
      int k = 0;
      for (i64 i = 0; i < p->D; ++i) {
        i64 d = p->dur[i];
        if (t - d < 0) continue;
        if (d > 0) { /* blank arc (t-d,u) -> (t,u) */
          i64 src = node_id(p, b, t - d, u);
          terms[k++] = alpha[src] + w_blank(p, tb, src, i);
        }
        if (u >= 1) { /* label arc (t-d,u-1) -> (t,u); d = 0 stays in frame t */
          i64 src = node_id(p, b, t - d, u - 1);
          terms[k++] = alpha[src] + w_label(p, tb, src, i);
        }
      }
      alpha[n] = log_sum_exp(terms, k);
    }
  }
  /* termination: a blank arc from (T_b - d, U_b) lands exactly on T_b */
  int k = 0;
  for (i64 i = 0; i < p->D; ++i) {
    i64 d = p->dur[i];
    if (d > 0 && Tb - d >= 0) {
      i64 src = node_id(p, b, Tb - d, Ub);
      terms[k++] = alpha[src] + w_blank(p, tb, src, i);
    }
  }
  double ll = log_sum_exp(terms, k);
  free(terms);
  return ll;
}

/* Backward variables: beta(t,u) = log of the summed weight of all path
 * suffixes from (t,u) to the end.  Returns beta(0,0). */
static double run_beta(const problem *p, const tables *tb, i64 b, double *beta) {
  i64 Tb = p->logit_lens[b], Ub = p->label_lens[b];
  double *terms = (double *)malloc(sizeof(double) * (size_t)(2 * p->D + 1));
  for (i64 t = Tb - 1; t >= 0; --t) {
    for (i64 u = Ub; u >= 0; --u) {
      i64 n = node_id(p, b, t, u);
      int k = 0;
      for (i64 i = 0; i < p->D; ++i) {
        i64 d = p->dur[i];
        if (d > 0) {
          if (t + d < Tb) terms[k++] = beta[node_id(p, b, t + d, u)] + w_blank(p, tb, n, i);
          else if (t + d == Tb && u == Ub) terms[k++] = w_blank(p, tb, n, i);
        }
        if (u < Ub && t + d < Tb)
          terms[k++] = beta[node_id(p, b, t + d, u + 1)] + w_label(p, tb, n, i);
      }
      beta[n] = log_sum_exp(terms, k);
    }
  }
  free(terms);
  return beta[node_id(p, b, 0, 0)];
}

/* Gradient of the reduced loss w.r.t. one logits row; zeros outside the
 * utterance's lattice and for utterances with no finite likelihood. */
static void grad_row(const problem *p, const tables *tb, const double *alpha, const double *beta,
                     const double *loglik, const double *scale, const int *valid, i64 n,
                     double *g) {
  for (i64 k = 0; k < p->VD; ++k) g[k] = 0.0;
  i64 b = n / (p->T * p->U1), t = (n / p->U1) % p->T, u = n % p->U1;
  if (!valid[b]) return;
  i64 Tb = p->logit_lens[b], Ub = p->label_lens[b];
  if (t >= Tb || u > Ub) return;
  double ll = loglik[b];
  if (!isfinite(ll)) return;
  double c = scale[b];
  double occ = exp(alpha[n] + beta[n] - ll); /* N(t,u): probability that a path visits (t,u) */
  if (alpha[n] == -INFINITY || beta[n] == -INFINITY) occ = 0.0;
  double gb_sum = 0.0, gl_sum = 0.0;
  double *gd = (double *)calloc((size_t)p->D, sizeof(double));
  for (i64 i = 0; i < p->D; ++i) {
    i64 d = p->dur[i];
    if (d > 0) {
      double bd = -INFINITY;
      if (t + d < Tb) bd = beta[node_id(p, b, t + d, u)];
      else if (t + d == Tb && u == Ub) bd = 0.0;
      double gam = (bd == -INFINITY || alpha[n] == -INFINITY)
                       ? 0.0
                       : exp(alpha[n] + w_blank(p, tb, n, i) + bd - ll);
      gb_sum += gam;
      gd[i] += gam;
    }
    if (u < Ub && t + d < Tb) {
      double bd = beta[node_id(p, b, t + d, u + 1)];
      double gam = (bd == -INFINITY || alpha[n] == -INFINITY)
                       ? 0.0
                       : exp(alpha[n] + w_label(p, tb, n, i) + bd - ll);
      gl_sum += gam;
      gd[i] += gam;
    }
  }
  i64 y = (u < Ub) ? p->labels[b * p->labels_stride + u] : -1;
  for (i64 k = 0; k < p->V; ++k) {
    double sm = exp(z_at(p, b, t, u, k) - tb->lse_tok[n]);
    double v = sm * occ;
    if (k == p->blank) v -= gb_sum;
    if (k == y) v -= gl_sum;
    g[k] = c * v;
  }
  for (i64 i = 0; i < p->D; ++i) {
    double smd = exp(tb->lp_dur[n * p->D + i]);
    g[p->V + i] = c * (smd * occ - gd[i]);
  }
  free(gd);
}

/*
 * Full evaluation.  Shapes: logits [B,T,U1,V+D] addressed with element
 * strides (any layout, e.g. a slice of a wider tensor); labels [B, >=U1-1]
 * with labels_stride elements per utterance; lengths [B].
 * Outputs (each may be NULL):
 *   loss_out  [B] for reduction none, else [1]
 *   utt_loss  [B]      per-utterance L_b (NaN for an unusable utterance)
 *   scale     [B]      c_b, the factor of dL_b/dz in the reduced loss
 *   alpha, beta [B*T*U1]  lattice variables (NaN outside the lattice)
 *   ll_alpha, ll_beta [B] log-likelihood from alpha and beta(0,0)
 *   grad      [n_rows][V+D] for the flat node ids in rows, or all
 *             B*T*U1 rows when rows == NULL
 */
int tdt_oracle_run(const void *logits, int logits_f64, const i64 *sizes, const i64 *strides,
                   const i64 *labels, i64 labels_stride, const i64 *logit_lens,
                   const i64 *label_lens, const int *durations, int n_dur, int blank,
                   double sigma, int reduction, double *loss_out, double *utt_loss,
                   double *scale_out, double *alpha_out, double *beta_out, double *ll_alpha,
                   double *ll_beta, const i64 *rows, i64 n_rows, double *grad) {
  if (!logits || !sizes || !strides || !labels || !logit_lens || !label_lens || !durations)
    return OR_EINVAL;
  problem p;
  p.logits = logits;
  p.logits_f64 = logits_f64;
  p.B = sizes[0]; p.T = sizes[1]; p.U1 = sizes[2]; p.VD = sizes[3];
  p.D = n_dur; p.V = p.VD - p.D;
  p.s0 = strides[0]; p.s1 = strides[1]; p.s2 = strides[2]; p.s3 = strides[3];
  p.labels = labels; p.labels_stride = labels_stride;
  p.logit_lens = logit_lens; p.label_lens = label_lens;
  p.dur = durations; p.blank = blank; p.sigma = sigma;
  if (p.B < 0 || p.T < 1 || p.U1 < 1 || n_dur < 1 || p.V < 1) return OR_EINVAL;
  if (blank < 0 || blank >= p.V) return OR_EINVAL;
  for (int i = 0; i < n_dur; ++i)
    if (durations[i] < 0) return OR_EINVAL;
  if (reduction < OR_RED_NONE || reduction > OR_RED_MEAN_VOLUME) return OR_EINVAL;

  i64 nodes = p.B * p.T * p.U1;
  int *valid = (int *)calloc((size_t)(p.B > 0 ? p.B : 1), sizeof(int));
  tables tb;
  tb.lse_tok = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes : 1));
  tb.lp_blank = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes : 1));
  tb.lp_label = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes : 1));
  tb.lp_dur = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes * p.D : 1));
  double *alpha = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes : 1));
  double *beta = (double *)malloc(sizeof(double) * (size_t)(nodes > 0 ? nodes : 1));
  double *lla = (double *)malloc(sizeof(double) * (size_t)(p.B > 0 ? p.B : 1));
  double *llb = (double *)malloc(sizeof(double) * (size_t)(p.B > 0 ? p.B : 1));
  double *lb = (double *)malloc(sizeof(double) * (size_t)(p.B > 0 ? p.B : 1));
  double *cb = (double *)malloc(sizeof(double) * (size_t)(p.B > 0 ? p.B : 1));
  if (!valid || !tb.lse_tok || !tb.lp_blank || !tb.lp_label || !tb.lp_dur || !alpha || !beta ||
      !lla || !llb || !lb || !cb) {
    free(valid); free(tb.lse_tok); free(tb.lp_blank); free(tb.lp_label); free(tb.lp_dur);
    free(alpha); free(beta); free(lla); free(llb); free(lb); free(cb);
    return OR_ENOMEM;
  }
  for (i64 b = 0; b < p.B; ++b) valid[b] = utterance_valid(&p, b);
  build_tables(&p, valid, &tb);
  for (i64 n = 0; n < nodes; ++n) { alpha[n] = NAN; beta[n] = NAN; }

#pragma omp parallel for schedule(dynamic, 1)
  for (i64 b = 0; b < p.B; ++b) {
    if (!valid[b]) { lla[b] = NAN; llb[b] = NAN; continue; }
    lla[b] = run_alpha(&p, &tb, b, alpha);
    llb[b] = run_beta(&p, &tb, b, beta);
  }

  /* L_b and the reduction (plain readings of the five names):
   *   none        loss[b] = L_b                    c_b = 1
   *   sum         sum_b L_b                        c_b = 1
   *   mean        (1/B) sum_b L_b / U_b            c_b = 1 / (B U_b)
   *   mean_batch  (1/B) sum_b L_b                  c_b = 1 / B
   *   mean_volume sum_b L_b / sum_b U_b            c_b = 1 / sum_b U_b   */
  double sum_u = 0.0;
  for (i64 b = 0; b < p.B; ++b) sum_u += (double)label_lens[b];
  for (i64 b = 0; b < p.B; ++b) {
    lb[b] = valid[b] ? -lla[b] : NAN;
    switch (reduction) {
      case OR_RED_MEAN: cb[b] = 1.0 / ((double)p.B * (double)label_lens[b]); break;
      case OR_RED_MEAN_BATCH: cb[b] = 1.0 / (double)p.B; break;
      case OR_RED_MEAN_VOLUME: cb[b] = 1.0 / sum_u; break;
      default: cb[b] = 1.0; break;
    }
  }
  if (loss_out) {
    if (reduction == OR_RED_NONE) {
      for (i64 b = 0; b < p.B; ++b) loss_out[b] = lb[b];
    } else {
      double acc = 0.0;
      for (i64 b = 0; b < p.B; ++b)
        acc += (reduction == OR_RED_MEAN) ? lb[b] / (double)label_lens[b] : lb[b];
      if (reduction == OR_RED_MEAN || reduction == OR_RED_MEAN_BATCH) acc /= (double)p.B;
      if (reduction == OR_RED_MEAN_VOLUME) acc /= sum_u;
      loss_out[0] = acc;
    }
  }
  if (utt_loss) memcpy(utt_loss, lb, sizeof(double) * (size_t)p.B);
  if (scale_out) memcpy(scale_out, cb, sizeof(double) * (size_t)p.B);
  if (alpha_out) memcpy(alpha_out, alpha, sizeof(double) * (size_t)nodes);
  if (beta_out) memcpy(beta_out, beta, sizeof(double) * (size_t)nodes);
  if (ll_alpha) memcpy(ll_alpha, lla, sizeof(double) * (size_t)p.B);
  if (ll_beta) memcpy(ll_beta, llb, sizeof(double) * (size_t)p.B);

  if (grad) {
    i64 nr = rows ? n_rows : nodes;
    int bad = 0;
    if (rows)
      for (i64 r = 0; r < nr; ++r)
        if (rows[r] < 0 || rows[r] >= nodes) bad = 1;
    if (!bad) {
#pragma omp parallel for schedule(static)
      for (i64 r = 0; r < nr; ++r)
        grad_row(&p, &tb, alpha, beta, lla, cb, valid, rows ? rows[r] : r, grad + r * p.VD);
    }
    if (bad) {
      free(valid); free(tb.lse_tok); free(tb.lp_blank); free(tb.lp_label); free(tb.lp_dur);
      free(alpha); free(beta); free(lla); free(llb); free(lb); free(cb);
      return OR_EINVAL;
    }
  }
  free(valid); free(tb.lse_tok); free(tb.lp_blank); free(tb.lp_label); free(tb.lp_dur);
  free(alpha); free(beta); free(lla); free(llb); free(lb); free(cb);
  return OR_OK;
}

/* Per-node log-softmax tables alone (for pinning the first step). Each
 * output is [B*T*U1] (lp_dur: [B*T*U1][D]); NaN outside the lattice. */
int tdt_oracle_tables(const void *logits, int logits_f64, const i64 *sizes, const i64 *strides,
                      const i64 *labels, i64 labels_stride, const i64 *logit_lens,
                      const i64 *label_lens, int n_dur, int blank, double *lse_tok,
                      double *lp_blank, double *lp_label, double *lp_dur) {
  problem p;
  memset(&p, 0, sizeof p);
  p.logits = logits;
  p.logits_f64 = logits_f64;
  p.B = sizes[0]; p.T = sizes[1]; p.U1 = sizes[2]; p.VD = sizes[3];
  p.D = n_dur; p.V = p.VD - p.D;
  p.s0 = strides[0]; p.s1 = strides[1]; p.s2 = strides[2]; p.s3 = strides[3];
  p.labels = labels; p.labels_stride = labels_stride;
  p.logit_lens = logit_lens; p.label_lens = label_lens;
  p.blank = blank;
  if (p.V < 1 || blank < 0 || blank >= p.V || n_dur < 1) return OR_EINVAL;
  int *valid = (int *)calloc((size_t)(p.B > 0 ? p.B : 1), sizeof(int));
  if (!valid) return OR_ENOMEM;
  for (i64 b = 0; b < p.B; ++b) valid[b] = utterance_valid(&p, b);
  tables tb = {lse_tok, lp_blank, lp_label, lp_dur};
  build_tables(&p, valid, &tb);
  free(valid);
  return OR_OK;
}
