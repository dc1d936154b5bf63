// tdt_grad.cu -- K4: the fused gradient pass over all V+D logits of a node.
//
// "one fused kernel for the gradients w.r.t. the token and duration logits"
// ("tdt-loss: add TDT loss kernel", kernels-community PR #882, "What's in
// it").  With N = exp(alpha + beta - logL) the occupancy of node (t,u), and
// fB, fL, fD_i the shares of beta(t,u) through its blank arcs, its label
// arcs and each duration (so N fB = sum of blank-arc posteriors, etc.):
//   dL/dz_k     = c_b N (softmax_k - [k = blank] fB - [k = y_{u+1}] fL),  k < V
//   dL/dz_{V+i} = c_b N (softmaxD_i - fD_i)
// The softmaxes are recomputed from the row and the saved log-sum-exps, so
// the row is read once more and every gradient element written once, in the
// input dtype (round to nearest).  Rows outside a lattice are written as 0.
// One warp per row; 16-byte loads and stores when the input row and the
// output row have the same offset from a 16-byte boundary (the contiguous
// case), coalesced scalar accesses otherwise.
#include "tdt_rowio.cuh"

namespace tdt {

namespace {

constexpr int kGradThreads = 256;
constexpr int kGradUnroll = 4;
constexpr int kScalarUnroll = 8;

template <int DT>
__device__ __forceinline__ void zero_row(typename Elem<DT>::T *out, long long VD, int lane) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  int head = head_elems<DT>(out);
  if (head > VD) head = (int)VD;
  const long long nvec = (VD - head) / N;
  const long long tail0 = head + nvec * N;
  const E zero = Elem<DT>::from_float(0.0f);
  if (lane < head) out[lane] = zero;
  if (lane < VD - tail0) out[tail0 + lane] = zero;
  uint4 *v = reinterpret_cast<uint4 *>(out + head);
  for (long long j = lane; j < nvec; j += 32) v[j] = make_uint4(0u, 0u, 0u, 0u);
}

template <int DT>
__global__ void __launch_bounds__(kGradThreads)
grad_kernel(Problem p, Workspace ws, typename Elem<DT>::T *grad, long long n_begin,
            long long n_end) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  const E *logits = static_cast<const E *>(p.logits);
  const int lane = threadIdx.x & 31;
  const long long n = n_begin + (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (n >= n_end) return;
  const long long nodes = p.B * p.T * p.U1;
  const long long u = n % p.U1;
  const long long bt = n / p.U1;
  const long long t = bt % p.T;
  const long long b = bt / p.T;
  E *out = grad + n * p.VD;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  bool live = ws.usable[b] && t < Tb && u <= Ub;
  float a = 0.0f;
  if (live) {
    // N = exp(alpha + beta - logL) = 2^((m_a + m_b - m_L) log2 e) * s_a * s_b / s_L
    const long long q = diag_index(p, b, t, u);
    const LV al = ws.alpha[q], be = ws.beta[q], ll = ws.loglik[b];
    if (al.s == 0.0f || be.s == 0.0f || ll.s == 0.0f) {
      live = false;
    } else {
      const fx_t dm = al.m + be.m - ll.m;
      const float occ = fast_exp2(__ll2float_rn(dm) * kFxToLog2) * (al.s * be.s / ll.s);
      a = (float)ws.scale[b] * occ;
    }
  }
  if (!live) {
    zero_row<DT>(out, p.VD, lane);
    return;
  }
  const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;
  const float lse2 = ws.lse_tok[n] * kLog2e;
  const float lsed2 = ws.lse_dur[n] * kLog2e;
  const float ab = a * ws.frac[n];           // a * fB, taken off the blank entry
  const float al = a * ws.frac[nodes + n];   // a * fL, taken off the label entry
  const long long y = (u < Ub) ? p.labels[b * (p.U1 - 1) + u] : -1;
  auto g_at = [&](float x, long long k) {
    float g = a * fast_exp2(fmaf(x, kLog2e, -lse2));
    if (k == p.blank) g -= ab;
    if (k == y) g -= al;
    return g;
  };

  const uintptr_t ai = reinterpret_cast<uintptr_t>(row), ao = reinterpret_cast<uintptr_t>(out);
  if (((ai ^ ao) & 15) == 0) {
    int head = head_elems<DT>(row);
    if (head > p.V) head = (int)p.V;
    const long long nvec = (p.V - head) / N;
    const long long tail0 = head + nvec * N;
    const int ntail = (int)(p.V - tail0);
    if (lane < head) out[lane] = Elem<DT>::from_float(g_at(Elem<DT>::load(row + lane), lane));
    if (lane < ntail) {
      const long long k = tail0 + lane;
      out[k] = Elem<DT>::from_float(g_at(Elem<DT>::load(row + k), k));
    }
    const uint4 *vin = reinterpret_cast<const uint4 *>(row + head);
    uint4 *vout = reinterpret_cast<uint4 *>(out + head);
    const int nv = (int)nvec;
    // vectors holding the two special entries (or -1)
    const int jb = (p.blank >= head && p.blank < tail0) ? (int)((p.blank - head) / N) : -1;
    const int jy = (y >= head && y < tail0) ? (int)((y - head) / N) : -1;
    const int eb = (int)((p.blank - head) % N), ey = (int)((y - head) % N);
    // Two batches of kGradUnroll vectors per lane: the next batch is loaded
    // before the current one is computed and stored.
    uint4 cur[kGradUnroll], nxt[kGradUnroll];
#pragma unroll
    for (int k = 0; k < kGradUnroll; ++k) {
      const int j = k * 32 + lane;
      if (j < nv) cur[k] = __ldg(vin + j);
    }
    for (int j0 = 0; j0 < nv; j0 += 32 * kGradUnroll) {
      const int jn = j0 + 32 * kGradUnroll;
#pragma unroll
      for (int k = 0; k < kGradUnroll; ++k) {
        const int j = jn + k * 32 + lane;
        if (j < nv) nxt[k] = __ldg(vin + j);
      }
#pragma unroll
      for (int k = 0; k < kGradUnroll; ++k) {
        const int j = j0 + k * 32 + lane;
        if (j < nv) {
          float x[N];
          unpack<DT>(cur[k], x);
#pragma unroll
          for (int e = 0; e < N; ++e) x[e] = a * fast_exp2(fmaf(x[e], kLog2e, -lse2));
          if (j == jb) x[eb] -= ab;
          if (j == jy) x[ey] -= al;
          vout[j] = pack<DT>(x);
        }
        cur[k] = nxt[k];
      }
    }
  } else {
    for (long long k0 = 0; k0 < p.V; k0 += 32 * kScalarUnroll) {
      float x[kScalarUnroll];
#pragma unroll
      for (int j = 0; j < kScalarUnroll; ++j) {
        const long long k = k0 + j * 32 + lane;
        x[j] = (k < p.V) ? Elem<DT>::load(row + k) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kScalarUnroll; ++j) {
        const long long k = k0 + j * 32 + lane;
        if (k < p.V) out[k] = Elem<DT>::from_float(g_at(x[j], k));
      }
    }
  }
  if (lane < p.D) {
    const float zd = Elem<DT>::load(row + p.V + lane);
    const float g = fast_exp2(fmaf(zd, kLog2e, -lsed2)) - ws.frac[(long long)(2 + lane) * nodes + n];
    out[p.V + lane] = Elem<DT>::from_float(a * g);
  }
}

}  // namespace

cudaError_t launch_grad(const Problem &p, int dtype, const Workspace &ws, void *grad_out,
                        long long n_begin, long long n_end, cudaStream_t stream) {
  const long long rows = n_end - n_begin;
  if (rows <= 0) return cudaSuccess;
  const long long warps_per_block = kGradThreads / 32;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  dim3 grid((unsigned)blocks), block(kGradThreads);
  switch (dtype) {
    case kF32:
      grad_kernel<kF32><<<grid, block, 0, stream>>>(p, ws, static_cast<float *>(grad_out),
                                                    n_begin, n_end);
      break;
    case kF16:
      grad_kernel<kF16><<<grid, block, 0, stream>>>(p, ws, static_cast<__half *>(grad_out),
                                                    n_begin, n_end);
      break;
    default:
      grad_kernel<kBF16><<<grid, block, 0, stream>>>(
          p, ws, static_cast<__nv_bfloat16 *>(grad_out), n_begin, n_end);
      break;
  }
  return cudaGetLastError();
}

}  // namespace tdt
