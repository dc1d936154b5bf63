/*
 * rnnt_oracle.c -- plain CPU oracle for the RNN-T loss (a transducer with
 * no duration head) and its gradient, in float64.
 *
 * TEST INFRASTRUCTURE ONLY, like tdt_oracle.c: only the test-suite uses it;
 * the product library never loads it and shares no code with it.
 *
 * Source: "Add TDT loss kernel" (transformers PR #46048), commit list:
 * torchaudio's rnnt_loss "does not train duration head" -- the plain RNN-T
 * loss is the transducer loss without durations.  Its lattice (Graves 2012,
 * "Sequence Transduction with Recurrent Neural Networks"), written out:
 *   node (t,u), 0 <= t < T_b, 0 <= u <= U_b;
 *   blank arc (t,u) -> (t+1,u),   weight lpB(t,u) - sigma;
 *   label arc (t,u) -> (t,u+1),   u < U_b, weight lpL(t,u) - sigma,
 *             lpL = log-softmax of label y_{u+1} = labels[b,u];
 *   a path starts at (0,0) and ends with the blank arc from (T_b-1, U_b).
 *   lpB, lpL: log-softmax over the V logits z[0..V) (blank inside).
 * sigma is kept as in the TDT loss (subtracted once per arc; 0 = plain
 * RNN-T).  Lengths, labels, reductions and unusable utterances follow the
 * same readings as tdt_oracle.c.
 *
 *   alpha(0,0) = 0
 *   alpha(t,u) = logaddexp(alpha(t-1,u) + wB(t-1,u), alpha(t,u-1) + wL(t,u-1))
 *   logL       = alpha(T_b-1, U_b) + wB(T_b-1, U_b)
 *   beta(T_b-1,U_b) = wB(T_b-1,U_b)
 *   beta(t,u)  = logaddexp(beta(t+1,u) + wB(t,u), beta(t,u+1) + wL(t,u))
 *   dL/dz_k(t,u) = c_b (softmax_k N - [k = blank] gB - [k = y_{u+1}] gL)
 *     N  = exp(alpha + beta - logL)                       occupancy of (t,u)
 *     gB = exp(alpha(t,u) + wB(t,u) + beta(t+1,u) - logL)  (beta(T_b,U_b) = 0)
 *     gL = exp(alpha(t,u) + wL(t,u) + beta(t,u+1) - logL)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int64_t r64;

static double lae(double a, double b) {  /* log(exp(a) + exp(b)) */
  if (a == -INFINITY) return b;
  if (b == -INFINITY) return a;
  double m = a > b ? a : b;
  return m + log(exp(a - m) + exp(b - m));
}

typedef struct {
  const void *logits;
  int f64;
  r64 B, T, U1, V;
  r64 s0, s1, s2, s3;
  const r64 *labels;
  r64 lstride;
  const r64 *tl, *ul;
  int blank;
  double sigma;
} rproblem;

static double rz(const rproblem *p, r64 b, r64 t, r64 u, r64 k) {
  r64 off = b * p->s0 + t * p->s1 + u * p->s2 + k * p->s3;
  return p->f64 ? ((const double *)p->logits)[off] : (double)((const float *)p->logits)[off];
}
static r64 rid(const rproblem *p, r64 b, r64 t, r64 u) { return (b * p->T + t) * p->U1 + u; }

static int rvalid(const rproblem *p, r64 b) {
  r64 Tb = p->tl[b], Ub = p->ul[b];
  if (Tb < 1 || Tb > p->T || Ub < 0 || Ub > p->U1 - 1) return 0;
  for (r64 u = 0; u < Ub; ++u) {
    r64 y = p->labels[b * p->lstride + u];
    if (y < 0 || y >= p->V || y == p->blank) return 0;
  }
  return 1;
}

/* log-sum-exp of the V logits of node (b,t,u) */
static double rlse(const rproblem *p, r64 b, r64 t, r64 u) {
  double m = -INFINITY;
  for (r64 k = 0; k < p->V; ++k) {
    double z = rz(p, b, t, u, k);
    if (z > m) m = z;
  }
  double s = 0.0;
  for (r64 k = 0; k < p->V; ++k) s += exp(rz(p, b, t, u, k) - m);
  return m + log(s);
}

/*
 * Outputs as tdt_oracle_run: loss_out ([B] for none, else [1]), utt_loss,
 * scale, alpha/beta [B*T*U1] (NaN outside lattices), ll_alpha/ll_beta [B],
 * grad [B*T*U1][V] (or NULL).  sizes = {B, T, U+1, V}.
 */
int rnnt_oracle_run(const void *logits, int logits_f64, const r64 *sizes, const r64 *strides,
                    const r64 *labels, r64 labels_stride, const r64 *logit_lens,
                    const r64 *label_lens, int blank, double sigma, int reduction,
                    double *loss_out, double *utt_loss, double *scale_out, double *alpha_out,
                    double *beta_out, double *ll_alpha, double *ll_beta, double *grad) {
  if (!logits || !sizes || !strides || !logit_lens || !label_lens) return -1;
  rproblem p;
  p.logits = logits; p.f64 = logits_f64;
  p.B = sizes[0]; p.T = sizes[1]; p.U1 = sizes[2]; p.V = sizes[3];
  p.s0 = strides[0]; p.s1 = strides[1]; p.s2 = strides[2]; p.s3 = strides[3];
  p.labels = labels; p.lstride = labels_stride;
  p.tl = logit_lens; p.ul = label_lens; p.blank = blank; p.sigma = sigma;
  if (p.B < 0 || p.T < 1 || p.U1 < 1 || p.V < 1 || blank < 0 || blank >= p.V) return -1;
  if (reduction < 0 || reduction > 4) return -1;
  if (p.U1 > 1 && !labels) return -1;
  const r64 nodes = p.B * p.T * p.U1;
  const size_t nn = (size_t)(nodes > 0 ? nodes : 1), nb = (size_t)(p.B > 0 ? p.B : 1);
  double *lse = malloc(sizeof(double) * nn), *wb = malloc(sizeof(double) * nn);
  double *wl = malloc(sizeof(double) * nn), *al = malloc(sizeof(double) * nn);
  double *be = malloc(sizeof(double) * nn), *lla = malloc(sizeof(double) * nb);
  double *llb = malloc(sizeof(double) * nb), *lb = malloc(sizeof(double) * nb);
  double *cb = malloc(sizeof(double) * nb);
  int *valid = calloc(nb, sizeof(int));
  if (!lse || !wb || !wl || !al || !be || !lla || !llb || !lb || !cb || !valid) {
    free(lse); free(wb); free(wl); free(al); free(be); free(lla); free(llb); free(lb);
    free(cb); free(valid);
    return -2;
  }
  for (r64 b = 0; b < p.B; ++b) valid[b] = rvalid(&p, b);
  for (r64 n = 0; n < nodes; ++n) {
    lse[n] = wb[n] = wl[n] = al[n] = be[n] = NAN;
  }

#pragma omp parallel for schedule(dynamic, 1)
  for (r64 b = 0; b < p.B; ++b) {
    if (!valid[b]) { lla[b] = llb[b] = NAN; continue; }
    const r64 Tb = p.tl[b], Ub = p.ul[b];
    for (r64 t = 0; t < Tb; ++t)
      for (r64 u = 0; u <= Ub; ++u) {
        const r64 n = rid(&p, b, t, u);
        lse[n] = rlse(&p, b, t, u);
        wb[n] = rz(&p, b, t, u, blank) - lse[n] - sigma;
        wl[n] = -INFINITY;
        if (u < Ub) wl[n] = rz(&p, b, t, u, labels[b * labels_stride + u]) - lse[n] - sigma;
      }
    for (r64 t = 0; t < Tb; ++t)
      for (r64 u = 0; u <= Ub; ++u) {
        const r64 n = rid(&p, b, t, u);
        if (t == 0 && u == 0) { al[n] = 0.0; continue; }
        double a = -INFINITY;
        if (t >= 1) a = lae(a, al[rid(&p, b, t - 1, u)] + wb[rid(&p, b, t - 1, u)]);
        if (u >= 1) a = lae(a, al[rid(&p, b, t, u - 1)] + wl[rid(&p, b, t, u - 1)]);
        al[n] = a;
      }
    lla[b] = al[rid(&p, b, Tb - 1, Ub)] + wb[rid(&p, b, Tb - 1, Ub)];
    for (r64 t = Tb - 1; t >= 0; --t)
      for (r64 u = Ub; u >= 0; --u) {
        const r64 n = rid(&p, b, t, u);
        if (t == Tb - 1 && u == Ub) { be[n] = wb[n]; continue; }
        double v = -INFINITY;
        if (t + 1 < Tb) v = lae(v, be[rid(&p, b, t + 1, u)] + wb[n]);
        if (u < Ub) v = lae(v, be[rid(&p, b, t, u + 1)] + wl[n]);
        be[n] = v;
      }
    llb[b] = be[rid(&p, b, 0, 0)];
  }

  double sum_u = 0.0;
  for (r64 b = 0; b < p.B; ++b) sum_u += (double)label_lens[b];
  for (r64 b = 0; b < p.B; ++b) {
    lb[b] = valid[b] ? -lla[b] : NAN;
    cb[b] = reduction == 2 ? 1.0 / ((double)p.B * (double)label_lens[b])
          : reduction == 3 ? 1.0 / (double)p.B
          : reduction == 4 ? 1.0 / sum_u : 1.0;
  }
  if (loss_out) {
    if (reduction == 0) {
      for (r64 b = 0; b < p.B; ++b) loss_out[b] = lb[b];
    } else {
      double acc = 0.0;
      for (r64 b = 0; b < p.B; ++b) acc += reduction == 2 ? lb[b] / (double)label_lens[b] : lb[b];
      if (reduction == 2 || reduction == 3) acc /= (double)p.B;
      if (reduction == 4) acc /= sum_u;
      loss_out[0] = acc;
    }
  }
  if (utt_loss) memcpy(utt_loss, lb, sizeof(double) * (size_t)p.B);
  if (scale_out) memcpy(scale_out, cb, sizeof(double) * (size_t)p.B);
  if (alpha_out) memcpy(alpha_out, al, sizeof(double) * (size_t)nodes);
  if (beta_out) memcpy(beta_out, be, sizeof(double) * (size_t)nodes);
  if (ll_alpha) memcpy(ll_alpha, lla, sizeof(double) * (size_t)p.B);
  if (ll_beta) memcpy(ll_beta, llb, sizeof(double) * (size_t)p.B);

  if (grad) {
#pragma omp parallel for schedule(static)
    for (r64 n = 0; n < nodes; ++n) {
      double *g = grad + n * p.V;
      for (r64 k = 0; k < p.V; ++k) g[k] = 0.0;
      const r64 b = n / (p.T * p.U1), t = (n / p.U1) % p.T, u = n % p.U1;
      if (!valid[b] || t >= p.tl[b] || u > p.ul[b] || !isfinite(lla[b])) continue;
      const r64 Tb = p.tl[b], Ub = p.ul[b];
      const double ll = lla[b];
      const double occ = (al[n] == -INFINITY || be[n] == -INFINITY) ? 0.0
                         : exp(al[n] + be[n] - ll);
      double bnext = -INFINITY;  /* beta after the blank arc */
      if (t + 1 < Tb) bnext = be[rid(&p, b, t + 1, u)];
      else if (u == Ub) bnext = 0.0;
      const double gB = (al[n] == -INFINITY || bnext == -INFINITY) ? 0.0
                        : exp(al[n] + wb[n] + bnext - ll);
      double gL = 0.0;
      if (u < Ub && al[n] != -INFINITY && be[rid(&p, b, t, u + 1)] != -INFINITY)
        gL = exp(al[n] + wl[n] + be[rid(&p, b, t, u + 1)] - ll);
      const r64 y = u < Ub ? labels[b * labels_stride + u] : -1;
      for (r64 k = 0; k < p.V; ++k) {
        double v = exp(rz(&p, b, t, u, k) - lse[n]) * occ;
        if (k == blank) v -= gB;
        if (k == y) v -= gL;
        g[k] = cb[b] * v;
      }
    }
  }
  free(lse); free(wb); free(wl); free(al); free(be); free(lla); free(llb); free(lb);
  free(cb); free(valid);
  return 0;
}
