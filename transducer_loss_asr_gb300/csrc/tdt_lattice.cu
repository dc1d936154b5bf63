// tdt_lattice.cu -- K2 alpha, K3 beta (+ arc fractions), K5 reduction.
//
// "alpha/beta passes over the lattice (float64 accumulation for precision on
// long label sequences, no 1024-label limit)" ("tdt-loss: add TDT loss
// kernel", kernels-community PR #882, "What's in it").  alpha(t,u) depends on
// (t-d,u) for d > 0 and on (t-d,u-1) for every d including 0, so all of its
// inputs lie on earlier anti-diagonals t+u: one CTA per utterance walks the
// anti-diagonals in order, one thread per node of the current diagonal (as
// many nodes per thread as needed: no limit on U), with a CTA barrier
// between diagonals.  beta walks them in reverse.  Values are fx (64-bit
// fixed point, see tdt_common.cuh) and live in global memory in the
// anti-diagonal layout, so the reads of one diagonal step are contiguous.
#include "tdt_common.cuh"

namespace tdt {

namespace {

constexpr int kLatticeMaxThreads = 1024;

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
  for (long long j = threadIdx.x; j < p.B; j += blockDim.x) part += (unsigned long long)p.label_lens[j];
  atomicAdd(&s_sum, part);
  __syncthreads();
  const bool ok = s_ok != 0;
  *sum_u_out = (double)(long long)s_sum;
  __syncthreads();
  return ok;
}

__device__ __forceinline__ fx_t lpd_at(const Problem &p, const Workspace &ws, int i, long long q) {
  return ws.lpd[(long long)i * (p.B * p.n_diag * p.U1) + q];
}

// log-likelihood: a blank arc from (T_b - d, U_b) lands exactly on T_b.
// Reads alpha and the tables from global memory (one thread).
__device__ fx_t termination(const Problem &p, const Workspace &ws, long long b, long long Tb,
                            long long Ub) {
  fx_t m = kFxNegInf;
  for (int i = 0; i < p.n_dur; ++i) {
    const int d = p.dur[i];
    if (d <= 0 || Tb - d < 0) continue;
    const long long q = diag_index(p, b, Tb - d, Ub);
    const fx_t a = ws.alpha[q];
    if (a != kFxNegInf) m = fmax_fx(m, a + ws.wb[q] + lpd_at(p, ws, i, q));
  }
  if (m == kFxNegInf) return kFxNegInf;
  float sum = 0.0f;
  for (int i = 0; i < p.n_dur; ++i) {
    const int d = p.dur[i];
    if (d <= 0 || Tb - d < 0) continue;
    const long long q = diag_index(p, b, Tb - d, Ub);
    const fx_t a = ws.alpha[q];
    if (a != kFxNegInf)
      sum += fast_exp2(__ll2float_rn(a + ws.wb[q] + lpd_at(p, ws, i, q) - m) * kFxToLog2);
  }
  return m + fx_log_ge1(sum);
}

__global__ void __launch_bounds__(kLatticeMaxThreads)
alpha_kernel(Problem p, Workspace ws, long long b0) {
  const long long b = b0 + blockIdx.x;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (threadIdx.x == 0) {
    ws.usable[b] = ok ? 1 : 0;
    double c = 1.0;
    if (p.reduction == kMean) c = 1.0 / ((double)p.B * (double)p.label_lens[b]);
    else if (p.reduction == kMeanBatch) c = 1.0 / (double)p.B;
    else if (p.reduction == kMeanVolume) c = 1.0 / sum_u;
    ws.scale[b] = c;
  }
  if (!ok) {
    if (threadIdx.x == 0) ws.loglik[b] = kFxNegInf;
    return;
  }
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  for (long long s = 0; s < Tb + Ub; ++s) {
    const long long u_lo = s - (Tb - 1) > 0 ? s - (Tb - 1) : 0;
    const long long u_hi = s < Ub ? s : Ub;
    for (long long u = u_lo + threadIdx.x; u <= u_hi; u += blockDim.x) {
      const long long t = s - u;
      fx_t val = 0;
      if (s > 0) {
        fx_t m = kFxNegInf;
        for (int i = 0; i < p.n_dur; ++i) {
          const int d = p.dur[i];
          if (t - d < 0) continue;
          if (d > 0) {
            const long long q = diag_index(p, b, t - d, u);
            const fx_t a = ws.alpha[q];
            if (a != kFxNegInf) m = fmax_fx(m, a + ws.wb[q] + lpd_at(p, ws, i, q));
          }
          if (u >= 1) {
            const long long q = diag_index(p, b, t - d, u - 1);
            const fx_t a = ws.alpha[q];
            if (a != kFxNegInf) m = fmax_fx(m, a + ws.wl[q] + lpd_at(p, ws, i, q));
          }
        }
        if (m == kFxNegInf) {
          val = kFxNegInf;
        } else {
          float sum = 0.0f;
          for (int i = 0; i < p.n_dur; ++i) {
            const int d = p.dur[i];
            if (t - d < 0) continue;
            if (d > 0) {
              const long long q = diag_index(p, b, t - d, u);
              const fx_t a = ws.alpha[q];
              if (a != kFxNegInf)
                sum += fast_exp2(__ll2float_rn(a + ws.wb[q] + lpd_at(p, ws, i, q) - m) * kFxToLog2);
            }
            if (u >= 1) {
              const long long q = diag_index(p, b, t - d, u - 1);
              const fx_t a = ws.alpha[q];
              if (a != kFxNegInf)
                sum += fast_exp2(__ll2float_rn(a + ws.wl[q] + lpd_at(p, ws, i, q) - m) * kFxToLog2);
            }
          }
          val = m + fx_log_ge1(sum);
        }
      }
      ws.alpha[diag_index(p, b, t, u)] = val;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) ws.loglik[b] = termination(p, ws, b, Tb, Ub);
}

// beta(t,u) over the outgoing arcs of (t,u); also the share of beta(t,u)
// that goes through blank arcs, label arcs, and each duration (the arc
// posteriors divided by the node occupancy), for the gradient pass.
__global__ void __launch_bounds__(kLatticeMaxThreads)
beta_kernel(Problem p, Workspace ws, long long b0) {
  const long long b = b0 + blockIdx.x;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (!ok) return;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  const long long nodes = p.B * p.T * p.U1;
  for (long long s = Tb + Ub - 1; s >= 0; --s) {
    const long long u_lo = s - (Tb - 1) > 0 ? s - (Tb - 1) : 0;
    const long long u_hi = s < Ub ? s : Ub;
    for (long long u = u_lo + threadIdx.x; u <= u_hi; u += blockDim.x) {
      const long long t = s - u;
      const long long q = diag_index(p, b, t, u);
      const fx_t wb = ws.wb[q], wl = ws.wl[q];
      fx_t m = kFxNegInf;
      for (int i = 0; i < p.n_dur; ++i) {
        const int d = p.dur[i];
        const fx_t ld = lpd_at(p, ws, i, q);
        if (d > 0) {
          if (t + d < Tb) {
            const fx_t bb = ws.beta[diag_index(p, b, t + d, u)];
            if (bb != kFxNegInf) m = fmax_fx(m, bb + wb + ld);
          } else if (t + d == Tb && u == Ub) {
            m = fmax_fx(m, wb + ld);
          }
        }
        if (u < Ub && t + d < Tb) {
          const fx_t bb = ws.beta[diag_index(p, b, t + d, u + 1)];
          if (bb != kFxNegInf) m = fmax_fx(m, bb + wl + ld);
        }
      }
      const long long n = (b * p.T + t) * p.U1 + u;
      if (m == kFxNegInf) {
        ws.beta[q] = kFxNegInf;
        for (int k = 0; k < 2 + p.n_dur; ++k) ws.frac[(long long)k * nodes + n] = 0.0f;
        continue;
      }
      float sb = 0.0f, sl = 0.0f;
      for (int i = 0; i < p.n_dur; ++i) {
        const int d = p.dur[i];
        const fx_t ld = lpd_at(p, ws, i, q);
        float eb = 0.0f, el = 0.0f;
        if (d > 0) {
          if (t + d < Tb) {
            const fx_t bb = ws.beta[diag_index(p, b, t + d, u)];
            if (bb != kFxNegInf) eb = fast_exp2(__ll2float_rn(bb + wb + ld - m) * kFxToLog2);
          } else if (t + d == Tb && u == Ub) {
            eb = fast_exp2(__ll2float_rn(wb + ld - m) * kFxToLog2);
          }
        }
        if (u < Ub && t + d < Tb) {
          const fx_t bb = ws.beta[diag_index(p, b, t + d, u + 1)];
          if (bb != kFxNegInf) el = fast_exp2(__ll2float_rn(bb + wl + ld - m) * kFxToLog2);
        }
        sb += eb;
        sl += el;
        ws.frac[(long long)(2 + i) * nodes + n] = eb + el;  // normalised below
      }
      const float tot = sb + sl;
      const float inv = 1.0f / tot;
      ws.frac[n] = sb * inv;
      ws.frac[nodes + n] = sl * inv;
      for (int i = 0; i < p.n_dur; ++i) ws.frac[(long long)(2 + i) * nodes + n] *= inv;
      ws.beta[q] = m + fx_log_ge1(tot);
    }
    __syncthreads();
  }
}

// Per-utterance losses and the reduction into loss_out (float32).
__global__ void reduce_kernel(Problem p, Workspace ws, float *loss_out) {
  __shared__ double s_acc[32];
  __shared__ double s_vol[32];
  double acc = 0.0, vol = 0.0;
  for (long long b = threadIdx.x; b < p.B; b += blockDim.x) {
    double L;
    if (!ws.usable[b]) L = __longlong_as_double(0x7ff8000000000000LL);  // NaN
    else if (ws.loglik[b] == kFxNegInf) L = __longlong_as_double(0x7ff0000000000000LL);  // +inf
    else L = -(double)ws.loglik[b] / kFxOne;
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
  if (lane == 0) { s_acc[w] = acc; s_vol[w] = vol; }
  __syncthreads();
  if (threadIdx.x == 0 && p.reduction != kNone) {
    double a = 0.0, v = 0.0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) { a += s_acc[k]; v += s_vol[k]; }
    if (p.reduction == kMean || p.reduction == kMeanBatch) a /= (double)p.B;
    else if (p.reduction == kMeanVolume) a /= v;
    loss_out[0] = (float)a;
  }
}

int lattice_threads(const Problem &p) {
  long long th = ((p.U1 + 31) / 32) * 32;
  if (th > kLatticeMaxThreads) th = kLatticeMaxThreads;
  if (th < 32) th = 32;
  return (int)th;
}

// ---------------------------------------------------------------------------
// Shared-memory variant (U+1 <= 1024 and the rings fit in shared memory):
// thread u owns lattice row u.  alpha (or beta) of the last RA diagonals sits
// in a shared ring, and the per-node tables of the diagonals in flight in a
// second ring that cp.async fills kPrefetch diagonals ahead, so no global
// round trip sits on the step-to-step critical path.  blockIdx.y = 0 runs
// alpha, 1 runs beta (independent given the tables).

constexpr int kPrefetch = 6;

__device__ __forceinline__ void cp_async8(void *smem, const void *gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

struct Rings {
  fx_t *A;      // [RA][U1p]
  fx_t *W;      // [RW][F][U1p]: F = 2 + D fields (wb, wl, lpd[0..D-1])
  int mA, mW;   // RA - 1, RW - 1 (powers of two)
  int U1p, F;
  __device__ fx_t &a(long long q, int u) const { return A[(q & mA) * U1p + u]; }
  __device__ fx_t &w(long long q, int f, int u) const {
    return W[((q & mW) * F + f) * (long long)U1p + u];
  }
};

// Start the copies of diagonal q's table entries for this thread's node.
__device__ __forceinline__ void prefetch_diag(const Problem &p, const Workspace &ws,
                                              const Rings &r, long long b, long long q,
                                              long long Tb, long long Ub, int u) {
  const long long t = q - u;
  if (q >= 0 && u <= Ub && t >= 0 && t < Tb) {
    const long long gi = diag_index(p, b, t, u);
    const long long stride = p.B * p.n_diag * p.U1;
    cp_async8(&r.w(q, 0, u), ws.wb + gi);
    cp_async8(&r.w(q, 1, u), ws.wl + gi);
    for (int i = 0; i < p.n_dur; ++i) cp_async8(&r.w(q, 2 + i, u), ws.lpd + i * stride + gi);
  }
  cp_async_commit();
}

template <int MAXD>
__device__ void alpha_smem(const Problem &p, const Workspace &ws, const Rings &r, long long b,
                           long long Tb, long long Ub) {
  const int u = threadIdx.x;
  const long long nsteps = Tb + Ub;
  for (int k = 0; k < kPrefetch; ++k) prefetch_diag(p, ws, r, b, k, Tb, Ub, u);
  for (long long s = 0; s < nsteps; ++s) {
    prefetch_diag(p, ws, r, b, s + kPrefetch, Tb, Ub, u);
    cp_async_wait<kPrefetch>();
    __syncthreads();
    const long long t = s - u;
    if (u <= Ub && t >= 0 && t < Tb) {
      fx_t val = 0;
      if (s > 0) {
        fx_t c[2 * MAXD];
#pragma unroll
        for (int i = 0; i < MAXD; ++i) {
          fx_t cb = kFxNegInf, cl = kFxNegInf;
          if (i < p.n_dur) {
            const int d = p.dur[i];
            if (t - d >= 0) {
              if (d > 0) {
                const fx_t a = r.a(s - d, u);
                if (a != kFxNegInf) cb = a + r.w(s - d, 0, u) + r.w(s - d, 2 + i, u);
              }
              if (u >= 1) {
                const fx_t a = r.a(s - d - 1, u - 1);
                if (a != kFxNegInf) cl = a + r.w(s - d - 1, 1, u - 1) + r.w(s - d - 1, 2 + i, u - 1);
              }
            }
          }
          c[2 * i] = cb;
          c[2 * i + 1] = cl;
        }
        fx_t m = c[0];
#pragma unroll
        for (int k = 1; k < 2 * MAXD; ++k) m = fmax_fx(m, c[k]);
        if (m == kFxNegInf) {
          val = kFxNegInf;
        } else {
          float sum = 0.0f;
#pragma unroll
          for (int k = 0; k < 2 * MAXD; ++k)
            if (c[k] != kFxNegInf) sum += fast_exp2(__ll2float_rn(c[k] - m) * kFxToLog2);
          val = m + fx_log_ge1(sum);
        }
      }
      r.a(s, u) = val;
      ws.alpha[diag_index(p, b, t, u)] = val;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

template <int MAXD>
__device__ void beta_smem(const Problem &p, const Workspace &ws, const Rings &r, long long b,
                          long long Tb, long long Ub) {
  const int u = threadIdx.x;
  const long long last = Tb + Ub - 1;
  const long long nodes = p.B * p.T * p.U1;
  for (int k = 0; k < kPrefetch; ++k) prefetch_diag(p, ws, r, b, last - k, Tb, Ub, u);
  for (long long q = last; q >= 0; --q) {
    prefetch_diag(p, ws, r, b, q - kPrefetch, Tb, Ub, u);
    cp_async_wait<kPrefetch>();
    __syncthreads();
    const long long t = q - u;
    if (u <= Ub && t >= 0 && t < Tb) {
      const fx_t wb = r.w(q, 0, u), wl = r.w(q, 1, u);
      fx_t cb[MAXD], cl[MAXD];
#pragma unroll
      for (int i = 0; i < MAXD; ++i) {
        cb[i] = kFxNegInf;
        cl[i] = kFxNegInf;
        if (i < p.n_dur) {
          const int d = p.dur[i];
          const fx_t ld = r.w(q, 2 + i, u);
          if (d > 0) {
            if (t + d < Tb) {
              const fx_t bb = r.a(q + d, u);
              if (bb != kFxNegInf) cb[i] = bb + wb + ld;
            } else if (t + d == Tb && u == Ub) {
              cb[i] = wb + ld;
            }
          }
          if (u < Ub && t + d < Tb) {
            const fx_t bb = r.a(q + d + 1, u + 1);
            if (bb != kFxNegInf) cl[i] = bb + wl + ld;
          }
        }
      }
      fx_t m = kFxNegInf;
#pragma unroll
      for (int i = 0; i < MAXD; ++i) m = fmax_fx(m, fmax_fx(cb[i], cl[i]));
      const long long n = (b * p.T + t) * p.U1 + u;
      fx_t val = kFxNegInf;
      if (m == kFxNegInf) {
        for (int k = 0; k < 2 + p.n_dur; ++k) ws.frac[(long long)k * nodes + n] = 0.0f;
      } else {
        float eb[MAXD], el[MAXD], sb = 0.0f, sl = 0.0f;
#pragma unroll
        for (int i = 0; i < MAXD; ++i) {
          eb[i] = cb[i] != kFxNegInf ? fast_exp2(__ll2float_rn(cb[i] - m) * kFxToLog2) : 0.0f;
          el[i] = cl[i] != kFxNegInf ? fast_exp2(__ll2float_rn(cl[i] - m) * kFxToLog2) : 0.0f;
          sb += eb[i];
          sl += el[i];
        }
        const float tot = sb + sl;
        const float inv = 1.0f / tot;
        ws.frac[n] = sb * inv;
        ws.frac[nodes + n] = sl * inv;
#pragma unroll
        for (int i = 0; i < MAXD; ++i)
          if (i < p.n_dur) ws.frac[(long long)(2 + i) * nodes + n] = (eb[i] + el[i]) * inv;
        val = m + fx_log_ge1(tot);
      }
      r.a(q, u) = val;
      ws.beta[diag_index(p, b, t, u)] = val;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

template <int MAXD>
__global__ void __launch_bounds__(kLatticeMaxThreads)
lattice_smem_kernel(Problem p, Workspace ws, long long b0, int RA, int RW) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const long long b = b0 + blockIdx.x;
  const bool is_beta = blockIdx.y == 1;
  double sum_u;
  const bool ok = check_utterance(p, b, &sum_u);
  if (!is_beta && threadIdx.x == 0) {
    ws.usable[b] = ok ? 1 : 0;
    double c = 1.0;
    if (p.reduction == kMean) c = 1.0 / ((double)p.B * (double)p.label_lens[b]);
    else if (p.reduction == kMeanBatch) c = 1.0 / (double)p.B;
    else if (p.reduction == kMeanVolume) c = 1.0 / sum_u;
    ws.scale[b] = c;
    if (!ok) ws.loglik[b] = kFxNegInf;
  }
  if (!ok) return;
  Rings r;
  r.U1p = blockDim.x;
  r.F = 2 + p.n_dur;
  r.mA = RA - 1;
  r.mW = RW - 1;
  r.A = reinterpret_cast<fx_t *>(smem_raw);
  r.W = r.A + (long long)RA * r.U1p;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  if (!is_beta) {
    alpha_smem<MAXD>(p, ws, r, b, Tb, Ub);
    if (threadIdx.x == 0) ws.loglik[b] = termination(p, ws, b, Tb, Ub);
  } else {
    beta_smem<MAXD>(p, ws, r, b, Tb, Ub);
  }
}

int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

// Shared bytes of the ring variant, or 0 when it does not apply.
size_t smem_plan(const Problem &p, int *RA, int *RW, int *threads) {
  if (p.U1 > kLatticeMaxThreads || p.n_dur > 16) return 0;
  const int th = lattice_threads(p);
  const int ra = pow2_at_least(p.max_dur + 2);
  const int rw = pow2_at_least(kPrefetch + p.max_dur + 3);
  const size_t bytes = ((size_t)ra + (size_t)rw * (size_t)(2 + p.n_dur)) * (size_t)th * 8;
  if (bytes > 200 * 1024) return 0;
  *RA = ra;
  *RW = rw;
  *threads = th;
  return bytes;
}

}  // namespace

cudaError_t launch_lattice(const Problem &p, const Workspace &ws, long long b_begin,
                           long long b_end, bool with_beta, cudaStream_t stream) {
  const long long nb = b_end - b_begin;
  if (nb <= 0) return cudaSuccess;
  int RA = 0, RW = 0, th = 0;
  const size_t bytes = smem_plan(p, &RA, &RW, &th);
  if (bytes > 0) {
    dim3 grid((unsigned)nb, with_beta ? 2u : 1u);
    if (p.n_dur <= 8) {
      cudaFuncSetAttribute(lattice_smem_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes);
      lattice_smem_kernel<8><<<grid, th, bytes, stream>>>(p, ws, b_begin, RA, RW);
    } else {
      cudaFuncSetAttribute(lattice_smem_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes);
      lattice_smem_kernel<16><<<grid, th, bytes, stream>>>(p, ws, b_begin, RA, RW);
    }
    return cudaGetLastError();
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
