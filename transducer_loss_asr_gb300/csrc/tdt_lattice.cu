// tdt_lattice.cu -- K2 alpha, K3 beta (+ arc fractions), K5 reduction.
//
// "alpha/beta passes over the lattice (float64 accumulation for precision on
// long label sequences, no 1024-label limit)" ("tdt-loss: add TDT loss
// kernel", kernels-community PR #882, "What's in it").  alpha(t,u) depends on
// (t-d,u) for d > 0 and on (t-d,u-1) for every d including 0, so all of its
// inputs lie on earlier anti-diagonals t+u: one CTA per utterance and
// direction walks the anti-diagonals (in reverse for beta), one thread per
// node of the current diagonal, one barrier per diagonal.  Values are
// (m, s) pairs (tdt_common.cuh): exact 64-bit fixed point m plus an fp32
// mantissa s in [1, 2).  alpha and beta are also stored in global memory in
// the anti-diagonal layout for the gradient pass.
//
// Two variants:
//  * lattice_smem_kernel (U+1 <= 256, D <= 9, rings <= 200 KB): thread u
//    owns lattice row u; alpha/beta of the last RA diagonals sit in a shared
//    ring of 16-byte (m, s) records, and the arc-weight records of the
//    diagonals in flight in a second ring that cp.async fills kPrefetch
//    diagonals ahead, so no global round trip sits on the diagonal-to-
//    diagonal critical path.  Templated on the exact number of durations so
//    the arc loop is fully unrolled; all index arithmetic is 32-bit.
//  * alpha_kernel / beta_kernel: the same wavefront reading and writing
//    global memory, any U and D (no limit on label length).
#include "tdt_common.cuh"

namespace tdt {

namespace {

constexpr int kLatticeMaxThreads = 1024;
constexpr int kPrefetch = 6;
// Lanes per lattice node in the grouped shared-ring variant: 8 when a
// node's durations fit one per lane and the block fits, else 4.
constexpr int kGroupMax = 8;

__device__ __forceinline__ fx_t fmax_fx(fx_t a, fx_t b) { return a > b ? a : b; }

// Block-wide: are the lengths and the used labels of utterance b usable?
// Also returns sum_b U_b over the batch (for mean_volume).
__device__ bool check_utterance(const Problem &p, long long b, double *sum_u_out) {
  __shared__ int s_ok;
  __shared__ unsigned long long s_sum;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  if (threadIdx.x == 0) {
    s_ok = (Tb >= 1 && Tb <= p.T && Ub >= 0 && Ub <= p.U1 - 1) ? 1 : 0;
    s_sum = 0ull;
  }
  __syncthreads();
  if (s_ok) {
    for (long long u = threadIdx.x; u < Ub; u += blockDim.x) {
      const long long y = p.labels[b * (p.U1 - 1) + u];
      if (y < 0 || y >= p.V || y == p.blank) s_ok = 0;
    }
  }
  unsigned long long part = 0;
  for (long long j = threadIdx.x; j < p.B; j += blockDim.x)
    part += (unsigned long long)p.label_lens[j];
  atomicAdd(&s_sum, part);
  __syncthreads();
  const bool ok = s_ok != 0;
  *sum_u_out = (double)(long long)s_sum;
  __syncthreads();
  return ok;
}

// Per-utterance outputs of the alpha side: usable flag and c_b.
__device__ void write_utterance_info(const Problem &p, const Workspace &ws, long long b, bool ok,
                                     double sum_u) {
  ws.usable[b] = ok ? 1 : 0;
  double c = 1.0;
  if (p.reduction == kMean) c = 1.0 / ((double)p.B * (double)p.label_lens[b]);
  else if (p.reduction == kMeanBatch) c = 1.0 / (double)p.B;
  else if (p.reduction == kMeanVolume) c = 1.0 / sum_u;
  ws.scale[b] = c;
  if (!ok) {
    LV z;
    z.m = 0;
    z.s = 0.0f;
    z.pad = 0.0f;
    ws.loglik[b] = z;
  }
}

// Log-sum-exp of N candidate arcs (M_j, S_j) (S_j = 0: no arc) into (m, s);
// with TERMS also each arc's unnormalised term and 1 / their sum.
template <int N, bool TERMS>
__device__ __forceinline__ void lse_combine(const fx_t *M, const float *S, fx_t *m, float *s,
                                            float *term, float *inv_total) {
  fx_t ms = kFxNegInf;
#pragma unroll
  for (int j = 0; j < N; ++j)
    if (S[j] > 0.0f) ms = fmax_fx(ms, M[j]);
  if (ms == kFxNegInf) {
    *m = 0;
    *s = 0.0f;
    if (TERMS) {
#pragma unroll
      for (int j = 0; j < N; ++j) term[j] = 0.0f;
      *inv_total = 0.0f;
    }
    return;
  }
  float tot = 0.0f;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float e = 0.0f;
    if (S[j] > 0.0f) e = S[j] * fast_exp2(fx_diff_log2(M[j] - ms));
    if (TERMS) term[j] = e;
    tot += e;
  }
  lv_normalize(tot, ms, m, s);
  if (TERMS) *inv_total = fast_rcp(tot);
}

// Same for a runtime number of candidates (n <= 2 * kMaxDurations).
__device__ void lse_combine_n(const fx_t *M, const float *S, int n, fx_t *m, float *s,
                              float *term, float *inv_total) {
  fx_t ms = kFxNegInf;
  for (int j = 0; j < n; ++j)
    if (S[j] > 0.0f) ms = fmax_fx(ms, M[j]);
  if (ms == kFxNegInf) {
    *m = 0;
    *s = 0.0f;
    if (term)
      for (int j = 0; j < n; ++j) term[j] = 0.0f;
    if (inv_total) *inv_total = 0.0f;
    return;
  }
  float tot = 0.0f;
  for (int j = 0; j < n; ++j) {
    float e = 0.0f;
    if (S[j] > 0.0f) e = S[j] * fast_exp2(fx_diff_log2(M[j] - ms));
    if (term) term[j] = e;
    tot += e;
  }
  lv_normalize(tot, ms, m, s);
  if (inv_total) *inv_total = fast_rcp(tot);
}

__device__ __forceinline__ LV make_lv(fx_t m, float s) {
  LV v;
  v.m = m;
  v.s = s;
  v.pad = 0.0f;
  return v;
}

// log-likelihood: a blank arc from (T_b - d, U_b) lands exactly on T_b.
// Reads alpha and the arc weights from global memory (one thread).
__device__ void termination(const Problem &p, const Workspace &ws, long long b, long long Tb,
                            long long Ub) {
  fx_t M[kMaxDurations];
  float S[kMaxDurations];
  for (int i = 0; i < p.n_dur; ++i) {
    const int d = p.dur[i];
    M[i] = 0;
    S[i] = 0.0f;
    if (d <= 0 || Tb - d < 0) continue;
    const long long g = diag_index(p, b, Tb - d, Ub);
    const LV a = ws.alpha[g];
    S[i] = a.s;
    if (a.s > 0.0f) M[i] = a.m + ws.arcw[g * (2 * p.n_dur) + i];
  }
  fx_t m;
  float s;
  lse_combine_n(M, S, p.n_dur, &m, &s, nullptr, nullptr);
  ws.loglik[b] = make_lv(m, s);
}

// Shares of beta(t,u) through blank arcs, label arcs and each duration (arc
// posteriors divided by the node occupancy), from the per-arc terms.
__device__ __forceinline__ void write_fractions(const Problem &p, const Workspace &ws,
                                                long long n, const float *term, float inv,
                                                int nd) {
  const long long nodes = p.B * p.T * p.U1;
  float fb = 0.0f, fl = 0.0f;
  for (int i = 0; i < nd; ++i) {
    fb += term[i];
    fl += term[nd + i];
    ws.frac[(long long)(2 + i) * nodes + n] = (term[i] + term[nd + i]) * inv;
  }
  ws.frac[n] = fb * inv;
  ws.frac[nodes + n] = fl * inv;
}

// ---------------------------------------------------------------- fallback

__global__ void __launch_bounds__(kLatticeMaxThreads)
alpha_kernel(Problem p, Workspace ws, long long b0) {
  const long long b = b0 + blockIdx.x;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (threadIdx.x == 0) write_utterance_info(p, ws, b, ok, sum_u);
  if (!ok) return;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  const int nd = p.n_dur;
  for (long long s = 0; s < Tb + Ub; ++s) {
    const long long u_lo = s - (Tb - 1) > 0 ? s - (Tb - 1) : 0;
    const long long u_hi = s < Ub ? s : Ub;
    for (long long u = u_lo + threadIdx.x; u <= u_hi; u += blockDim.x) {
      const long long t = s - u;
      fx_t m = 0;
      float sv = 1.0f;
      if (s > 0) {
        fx_t M[2 * kMaxDurations];
        float S[2 * kMaxDurations];
        for (int i = 0; i < nd; ++i) {
          const int d = p.dur[i];
          M[i] = M[nd + i] = 0;
          S[i] = S[nd + i] = 0.0f;
          if (t - d < 0) continue;
          if (d > 0) {
            const long long g = diag_index(p, b, t - d, u);
            const LV a = ws.alpha[g];
            S[i] = a.s;
            if (a.s > 0.0f) M[i] = a.m + ws.arcw[g * (2 * nd) + i];
          }
          if (u >= 1) {
            const long long g = diag_index(p, b, t - d, u - 1);
            const LV a = ws.alpha[g];
            S[nd + i] = a.s;
            if (a.s > 0.0f) M[nd + i] = a.m + ws.arcw[g * (2 * nd) + nd + i];
          }
        }
        lse_combine_n(M, S, 2 * nd, &m, &sv, nullptr, nullptr);
      }
      ws.alpha[diag_index(p, b, t, u)] = make_lv(m, sv);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) termination(p, ws, b, Tb, Ub);
}

__global__ void __launch_bounds__(kLatticeMaxThreads)
beta_kernel(Problem p, Workspace ws, long long b0) {
  const long long b = b0 + blockIdx.x;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (!ok) return;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  const int nd = p.n_dur;
  for (long long s = Tb + Ub - 1; s >= 0; --s) {
    const long long u_lo = s - (Tb - 1) > 0 ? s - (Tb - 1) : 0;
    const long long u_hi = s < Ub ? s : Ub;
    for (long long u = u_lo + threadIdx.x; u <= u_hi; u += blockDim.x) {
      const long long t = s - u;
      const long long q = diag_index(p, b, t, u);
      const fx_t *rec = ws.arcw + q * (2 * nd);
      fx_t M[2 * kMaxDurations];
      float S[2 * kMaxDurations], term[2 * kMaxDurations];
      for (int i = 0; i < nd; ++i) {
        const int d = p.dur[i];
        M[i] = M[nd + i] = 0;
        S[i] = S[nd + i] = 0.0f;
        if (d > 0) {
          if (t + d < Tb) {
            const LV bb = ws.beta[diag_index(p, b, t + d, u)];
            S[i] = bb.s;
            if (bb.s > 0.0f) M[i] = bb.m + rec[i];
          } else if (t + d == Tb && u == Ub) {
            S[i] = 1.0f;
            M[i] = rec[i];
          }
        }
        if (u < Ub && t + d < Tb) {
          const LV bb = ws.beta[diag_index(p, b, t + d, u + 1)];
          S[nd + i] = bb.s;
          if (bb.s > 0.0f) M[nd + i] = bb.m + rec[nd + i];
        }
      }
      fx_t m;
      float sv, inv;
      lse_combine_n(M, S, 2 * nd, &m, &sv, term, &inv);
      write_fractions(p, ws, (b * p.T + t) * p.U1 + u, term, inv, nd);
      ws.beta[q] = make_lv(m, sv);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- shared-ring variant

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Shared rings of one CTA: A[RA][U1p] lattice values of the last RA
// diagonals; W[RW][U1p][2 ND] arc-weight records of the diagonals in flight.
template <int ND> struct Rings {
  LV *A;
  fx_t *W;
  int mA, mW, U1p;
  __device__ __forceinline__ LV &a(int q, int u) const { return A[(q & mA) * U1p + u]; }
  __device__ __forceinline__ const fx_t *w(int q, int u) const {
    return W + ((q & mW) * U1p + u) * (2 * ND);
  }
};

// Start the copies of diagonal q's record of node u (if it is a lattice
// node): lane k of the group copies the 16-byte chunks k, k+G, ...; every
// lane commits one group per call so the group count per step is fixed.
template <int ND, int G>
__device__ __forceinline__ void prefetch_group(const fx_t *gdiag0, const Rings<ND> &r, int q,
                                               int u, int k, int Tb, int Ub, int U1) {
  const int t = q - u;
  if (q >= 0 && u <= Ub && t >= 0 && t < Tb) {
    const fx_t *src = gdiag0 + ((long long)q * U1 + u) * (2 * ND);
    fx_t *dst = r.W + ((q & r.mW) * r.U1p + u) * (2 * ND);
    for (int c = k; c < ND; c += G) cp_async16(dst + 2 * c, src + 2 * c);
  }
  cp_async_commit();
}

// Grouped variant: lane k of a node's group of G lanes handles
// durations k, k+G, ... (both the blank and the label arc of each), so every
// lane runs the same instructions; the int64 max and the fp32 sum are
// combined across the group with xor shuffles.

template <int ND, int G>
struct GroupArcs {
  static constexpr int J = (ND + G - 1) / G;  // durations per lane
};

// Group-wide log-sum-exp of this lane's 2J candidates; returns the group's
// M* and S (S = 0 when the group has no finite candidate) and each
// candidate's unnormalised term.
template <int J, int G>
__device__ __forceinline__ void group_lse(const fx_t *M, const float *S, fx_t *ms_out,
                                          float *tot_out, float *term) {
  fx_t ms = M[0];
#pragma unroll
  for (int j = 1; j < 2 * J; ++j) ms = fmax_fx(ms, M[j]);
#pragma unroll
  for (int o = 1; o < G; o <<= 1) ms = fmax_fx(ms, __shfl_xor_sync(0xffffffffu, ms, o));
  float tot = 0.0f;
#pragma unroll
  for (int j = 0; j < 2 * J; ++j) {
    term[j] = S[j] * fast_exp2(fx_diff_log2_fast(M[j] - ms));
    tot += term[j];
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  *ms_out = ms;
  *tot_out = tot;
}

template <int ND, int G>
__device__ void alpha_grouped(const Problem &p, const Workspace &ws, const Rings<ND> &r,
                              long long b, int Tb, int Ub) {
  constexpr int J = GroupArcs<ND, G>::J;
  const int u = threadIdx.x / G, k = threadIdx.x % G;
  // node index for ring reads: threads past the last row (u >= U+1, in the
  // last warp) only join the barriers, and read row U1p - 1 so every read
  // stays in bounds
  const int uc = u < r.U1p ? u : r.U1p - 1;
  const int U1 = (int)p.U1;
  const fx_t *gdiag0 = ws.arcw + b * p.n_diag * p.U1 * (2 * ND);
  LV *galpha = ws.alpha + b * p.n_diag * p.U1;
  int di[J], dd[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    di[j] = k + G * j;
    dd[j] = di[j] < ND ? p.dur[di[j]] : -1;
  }
  const int nsteps = Tb + Ub;
  for (int q = 0; q < kPrefetch; ++q) prefetch_group<ND, G>(gdiag0, r, q, u, k, Tb, Ub, U1);
  for (int s = 0; s < nsteps; ++s) {
    prefetch_group<ND, G>(gdiag0, r, s + kPrefetch, u, k, Tb, Ub, U1);
    cp_async_wait<kPrefetch>();
    __syncthreads();
    const int t = s - u;
    const bool node = u <= Ub && t >= 0 && t < Tb;
    fx_t M[2 * J];
    float S[2 * J], term[2 * J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int d = dd[j];
      // blank arc (t-d, u) -> (t, u), d > 0
      const bool okb = node && d > 0 && t - d >= 0;
      const LV ab = r.a(s - d, uc);
      const fx_t wb = r.w(s - d, uc)[di[j] < ND ? di[j] : 0];
      M[2 * j] = okb ? ab.m + wb : kFxVeryNeg;
      S[2 * j] = okb ? ab.s : 0.0f;
      // label arc (t-d, u-1) -> (t, u), every d
      const bool okl = node && d >= 0 && u >= 1 && t - d >= 0;
      const int ul = uc >= 1 ? uc - 1 : 0;
      const LV al = r.a(s - d - 1, ul);
      const fx_t wl = r.w(s - d - 1, ul)[di[j] < ND ? ND + di[j] : 0];
      M[2 * j + 1] = okl ? al.m + wl : kFxVeryNeg;
      S[2 * j + 1] = okl ? al.s : 0.0f;
    }
    fx_t ms;
    float tot;
    group_lse<J, G>(M, S, &ms, &tot, term);
    if (node && k == 0) {
      LV v;
      if (s == 0) {
        v = make_lv(0, 1.0f);
      } else if (tot > 0.0f) {
        fx_t m;
        float sv;
        lv_normalize(tot, ms, &m, &sv);
        v = make_lv(m, sv);
      } else {
        v = make_lv(kFxVeryNeg, 0.0f);
      }
      r.a(s, u) = v;
      galpha[(long long)s * U1 + u] = v;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

template <int ND, int G>
__device__ void beta_grouped(const Problem &p, const Workspace &ws, const Rings<ND> &r,
                             long long b, int Tb, int Ub) {
  constexpr int J = GroupArcs<ND, G>::J;
  const int u = threadIdx.x / G, k = threadIdx.x % G;
  // node index for ring reads: threads past the last row (u >= U+1, in the
  // last warp) only join the barriers, and read row U1p - 1 so every read
  // stays in bounds
  const int uc = u < r.U1p ? u : r.U1p - 1;
  const int U1 = (int)p.U1;
  const fx_t *gdiag0 = ws.arcw + b * p.n_diag * p.U1 * (2 * ND);
  LV *gbeta = ws.beta + b * p.n_diag * p.U1;
  const long long nodes = p.B * p.T * p.U1;
  int di[J], dd[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    di[j] = k + G * j;
    dd[j] = di[j] < ND ? p.dur[di[j]] : -1;
  }
  const int last = Tb + Ub - 1;
  for (int i = 0; i < kPrefetch; ++i) prefetch_group<ND, G>(gdiag0, r, last - i, u, k, Tb, Ub, U1);
  for (int q = last; q >= 0; --q) {
    prefetch_group<ND, G>(gdiag0, r, q - kPrefetch, u, k, Tb, Ub, U1);
    cp_async_wait<kPrefetch>();
    __syncthreads();
    const int t = q - u;
    const bool node = u <= Ub && t >= 0 && t < Tb;
    const fx_t *rec = r.w(q, uc);
    fx_t M[2 * J];
    float S[2 * J], term[2 * J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int d = dd[j];
      const int i = di[j] < ND ? di[j] : 0;
      // blank arc (t, u) -> (t+d, u), d > 0; the final blank lands on T_b
      const bool inb = node && d > 0 && t + d < Tb;
      const bool fin = node && d > 0 && t + d == Tb && u == Ub;
      const LV bb = r.a(q + d, uc);
      M[2 * j] = inb ? bb.m + rec[i] : (fin ? rec[i] : kFxVeryNeg);
      S[2 * j] = inb ? bb.s : (fin ? 1.0f : 0.0f);
      // label arc (t, u) -> (t+d, u+1)
      const bool okl = node && d >= 0 && u < Ub && t + d < Tb;
      const LV bl = r.a(q + d + 1, uc + 1 < r.U1p ? uc + 1 : uc);
      M[2 * j + 1] = okl ? bl.m + rec[ND + i] : kFxVeryNeg;
      S[2 * j + 1] = okl ? bl.s : 0.0f;
    }
    fx_t ms;
    float tot;
    group_lse<J, G>(M, S, &ms, &tot, term);
    const float inv = tot > 0.0f ? fast_rcp(tot) : 0.0f;
    float fb = 0.0f, fl = 0.0f;
    const long long n = (b * p.T + t) * p.U1 + u;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      fb += term[2 * j];
      fl += term[2 * j + 1];
      if (node && di[j] < ND)
        ws.frac[(long long)(2 + di[j]) * nodes + n] = (term[2 * j] + term[2 * j + 1]) * inv;
    }
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
      fb += __shfl_xor_sync(0xffffffffu, fb, o);
      fl += __shfl_xor_sync(0xffffffffu, fl, o);
    }
    if (node && k == 0) {
      ws.frac[n] = fb * inv;
      ws.frac[nodes + n] = fl * inv;
      LV v;
      if (tot > 0.0f) {
        fx_t m;
        float sv;
        lv_normalize(tot, ms, &m, &sv);
        v = make_lv(m, sv);
      } else {
        v = make_lv(kFxVeryNeg, 0.0f);
      }
      r.a(q, u) = v;
      gbeta[(long long)q * U1 + u] = v;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

template <int ND, int G>
__global__ void __launch_bounds__(kLatticeMaxThreads, 1)
lattice_smem_kernel(Problem p, Workspace ws, long long b0, int RA, int RW) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const long long b = b0 + blockIdx.x;
  const bool is_beta = blockIdx.y == 1;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (!is_beta && threadIdx.x == 0) write_utterance_info(p, ws, b, ok, sum_u);
  if (!ok) return;
  Rings<ND> r;
  r.U1p = (int)p.U1;
  r.mA = RA - 1;
  r.mW = RW - 1;
  r.A = reinterpret_cast<LV *>(smem_raw);
  r.W = reinterpret_cast<fx_t *>(r.A + RA * r.U1p);
  const int Tb = (int)p.logit_lens[b], Ub = (int)p.label_lens[b];
  if (!is_beta) {
    alpha_grouped<ND, G>(p, ws, r, b, Tb, Ub);
    if (threadIdx.x == 0) termination(p, ws, b, Tb, Ub);
  } else {
    beta_grouped<ND, G>(p, ws, r, b, Tb, Ub);
  }
}

int lattice_threads(const Problem &p) {
  long long th = ((p.U1 + 31) / 32) * 32;
  if (th > kLatticeMaxThreads) th = kLatticeMaxThreads;
  if (th < 32) th = 32;
  return (int)th;
}

int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

// Shared bytes of the ring variant, or 0 when it does not apply.
int group_width(const Problem &p) {
  if (p.n_dur <= kGroupMax && p.U1 * kGroupMax <= kLatticeMaxThreads) return kGroupMax;
  return 4;
}

// Shared bytes of the ring variant (or 0 when it does not apply); threads =
// (U+1) * G rounded up to whole warps.
size_t smem_plan(const Problem &p, int *RA, int *RW, int *threads) {
  const int G = group_width(p);
  if (p.U1 * G > kLatticeMaxThreads || p.n_dur > 9) return 0;
  const int th = (int)(((p.U1 * G + 31) / 32) * 32);
  const int nodes_per_slot = (int)p.U1;
  const int ra = pow2_at_least(p.max_dur + 2);
  const int rw = pow2_at_least(kPrefetch + p.max_dur + 3);
  const size_t bytes =
      ((size_t)ra * sizeof(LV) + (size_t)rw * 16 * (size_t)p.n_dur) * (size_t)nodes_per_slot;
  if (bytes > 200 * 1024) return 0;
  *RA = ra;
  *RW = rw;
  *threads = th;
  return bytes;
}

template <int ND, int G>
cudaError_t launch_smem_g(const Problem &p, const Workspace &ws, long long b0, dim3 grid, int th,
                          size_t bytes, int RA, int RW, cudaStream_t stream) {
  // at least kLatticeSmemFloor, so no node-table or gradient block shares the SM
  if (bytes < (size_t)kLatticeSmemFloor) bytes = kLatticeSmemFloor;
  cudaError_t e = cudaFuncSetAttribute(lattice_smem_kernel<ND, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  lattice_smem_kernel<ND, G><<<grid, th, bytes, stream>>>(p, ws, b0, RA, RW);
  return cudaGetLastError();
}

template <int ND>
cudaError_t launch_smem(const Problem &p, const Workspace &ws, long long b0, dim3 grid, int th,
                        size_t bytes, int RA, int RW, cudaStream_t stream) {
  if (ND <= kGroupMax && group_width(p) == kGroupMax)
    return launch_smem_g<ND, kGroupMax>(p, ws, b0, grid, th, bytes, RA, RW, stream);
  return launch_smem_g<ND, 4>(p, ws, b0, grid, th, bytes, RA, RW, stream);
}

// ---------------------------------------------------------------- reduction

// Per-utterance losses and the reduction into loss_out (float32).
__global__ void reduce_kernel(Problem p, Workspace ws, float *loss_out) {
  __shared__ double s_acc[32];
  __shared__ double s_vol[32];
  double acc = 0.0, vol = 0.0;
  for (long long b = threadIdx.x; b < p.B; b += blockDim.x) {
    double L;
    if (!ws.usable[b]) L = __longlong_as_double(0x7ff8000000000000LL);                // NaN
    else if (ws.loglik[b].s == 0.0f) L = __longlong_as_double(0x7ff0000000000000LL);  // +inf
    else L = -((double)ws.loglik[b].m / kFxOne + log((double)ws.loglik[b].s));
    const double ub = (double)p.label_lens[b];
    if (p.reduction == kNone) loss_out[b] = (float)L;
    acc += (p.reduction == kMean) ? L / ub : L;
    vol += ub;
  }
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, o);
    vol += __shfl_xor_sync(0xffffffffu, vol, o);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_acc[w] = acc;
    s_vol[w] = vol;
  }
  __syncthreads();
  if (threadIdx.x == 0 && p.reduction != kNone) {
    double a = 0.0, v = 0.0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
      a += s_acc[k];
      v += s_vol[k];
    }
    if (p.reduction == kMean || p.reduction == kMeanBatch) a /= (double)p.B;
    else if (p.reduction == kMeanVolume) a /= v;
    loss_out[0] = (float)a;
  }
}

}  // namespace

cudaError_t launch_lattice(const Problem &p, const Workspace &ws, long long b_begin,
                           long long b_end, bool with_beta, cudaStream_t stream) {
  const long long nb = b_end - b_begin;
  if (nb <= 0) return cudaSuccess;
  int RA = 0, RW = 0, th = 0;
  const size_t bytes = smem_plan(p, &RA, &RW, &th);
  if (bytes > 0) {
    const dim3 grid((unsigned)nb, with_beta ? 2u : 1u);
    switch (p.n_dur) {
      case 1: return launch_smem<1>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 2: return launch_smem<2>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 3: return launch_smem<3>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 4: return launch_smem<4>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 5: return launch_smem<5>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 6: return launch_smem<6>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 7: return launch_smem<7>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      case 8: return launch_smem<8>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
      default: return launch_smem<9>(p, ws, b_begin, grid, th, bytes, RA, RW, stream);
    }
  }
  alpha_kernel<<<(unsigned)nb, lattice_threads(p), 0, stream>>>(p, ws, b_begin);
  if (with_beta) beta_kernel<<<(unsigned)nb, lattice_threads(p), 0, stream>>>(p, ws, b_begin);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const Problem &p, const Workspace &ws, float *loss_out,
                          cudaStream_t stream) {
  reduce_kernel<<<1, 256, 0, stream>>>(p, ws, loss_out);
  return cudaGetLastError();
}

}  // namespace tdt
