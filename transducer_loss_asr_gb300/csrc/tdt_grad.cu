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
#include "tdt_common.cuh"

namespace tdt {

namespace {

constexpr int kGradThreads = 256;
constexpr int kUnroll = 8;

template <int DT>
__global__ void __launch_bounds__(kGradThreads)
grad_kernel(Problem p, Workspace ws, typename Elem<DT>::T *grad) {
  typedef typename Elem<DT>::T E;
  const E *logits = static_cast<const E *>(p.logits);
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long nodes = p.B * p.T * p.U1;

  for (long long n = warp; n < nodes; n += nwarps) {
    const long long u = n % p.U1;
    const long long bt = n / p.U1;
    const long long t = bt % p.T;
    const long long b = bt / p.T;
    E *out = grad + n * p.VD;
    const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
    bool live = ws.usable[b] && t < Tb && u <= Ub && ws.loglik[b] != kFxNegInf;
    float a = 0.0f;
    if (live) {
      const long long q = diag_index(p, b, t, u);
      const fx_t al = ws.alpha[q], be = ws.beta[q];
      if (al == kFxNegInf || be == kFxNegInf) {
        live = false;
      } else {
        const float occ = fast_exp2(__ll2float_rn(al + be - ws.loglik[b]) * kFxToLog2);
        a = (float)ws.scale[b] * occ;
      }
    }
    if (!live) {
      const E zero = Elem<DT>::from_float(0.0f);
      for (long long k = lane; k < p.VD; k += 32) out[k] = zero;
      continue;
    }
    const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;
    const float lse_t = ws.lse_tok[n];
    const float lse_d = ws.lse_dur[n];
    const float fb = ws.frac[n];
    const float fl = ws.frac[nodes + n];
    const long long y = (u < Ub) ? p.labels[b * (p.U1 - 1) + u] : -1;
    for (long long k0 = 0; k0 < p.V; k0 += 32 * kUnroll) {
      float x[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const long long k = k0 + j * 32 + lane;
        x[j] = (k < p.V) ? Elem<DT>::load(row + k) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const long long k = k0 + j * 32 + lane;
        if (k < p.V) {
          float g = fast_exp2((x[j] - lse_t) * kLog2e);
          if (k == p.blank) g -= fb;
          if (k == y) g -= fl;
          out[k] = Elem<DT>::from_float(a * g);
        }
      }
    }
    if (lane < p.D) {
      const float zd = Elem<DT>::load(row + p.V + lane);
      const float g = fast_exp2((zd - lse_d) * kLog2e) - ws.frac[(long long)(2 + lane) * nodes + n];
      out[p.V + lane] = Elem<DT>::from_float(a * g);
    }
  }
}

}  // namespace

cudaError_t launch_grad(const Problem &p, int dtype, const Workspace &ws, void *grad_out,
                        cudaStream_t stream) {
  const long long nodes = p.B * p.T * p.U1;
  if (nodes == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long warps_per_block = kGradThreads / 32;
  long long blocks = (nodes + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  dim3 grid((unsigned)blocks), block(kGradThreads);
  switch (dtype) {
    case kF32:
      grad_kernel<kF32><<<grid, block, 0, stream>>>(p, ws, static_cast<float *>(grad_out));
      break;
    case kF16:
      grad_kernel<kF16><<<grid, block, 0, stream>>>(p, ws, static_cast<__half *>(grad_out));
      break;
    default:
      grad_kernel<kBF16><<<grid, block, 0, stream>>>(p, ws,
                                                     static_cast<__nv_bfloat16 *>(grad_out));
      break;
  }
  return cudaGetLastError();
}

}  // namespace tdt
