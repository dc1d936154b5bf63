// tdt_tables.cu -- K1: per-node log-softmax tables.
//
// "log-softmax over the vocabulary for each lattice node" ("tdt-loss: add
// TDT loss kernel", kernels-community PR #882, "What's in it"), plus the
// log-softmax of the duration logits.  One warp streams one logits row
// z[b,t,u,0:V+D) once, keeping a running max and a running sum of
// exp(z - max) per lane (fp32), then combines lanes with shuffles.  The row
// may be a slice of a wider tensor: only strides s0..s2 locate it.
//
// Outputs per usable node (t < T_b, u <= U_b):
//   lse_tok[n], lse_dur[n]         float, for the gradient pass
//   wb = lpB - sigma, wl = lpL - sigma, lpd[i]   fx, anti-diagonal layout,
//                                   for the alpha/beta passes
#include "tdt_common.cuh"

namespace tdt {

namespace {

constexpr int kTablesThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ fx_t clamp_lp(fx_t v) {
  const fx_t floor_fx = (fx_t)kLogProbFloor * (fx_t)4294967296LL;
  return v < floor_fx ? floor_fx : v;
}

template <int DT>
__global__ void __launch_bounds__(kTablesThreads)
node_tables_kernel(Problem p, Workspace ws) {
  typedef typename Elem<DT>::T E;
  const E *logits = static_cast<const E *>(p.logits);
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long nodes = p.B * p.T * p.U1;
  const long long ndiag_total = p.B * p.n_diag * p.U1;

  for (long long n = warp; n < nodes; n += nwarps) {
    const long long u = n % p.U1;
    const long long bt = n / p.U1;
    const long long t = bt % p.T;
    const long long b = bt / p.T;
    const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
    if (Tb < 1 || Tb > p.T || Ub < 0 || Ub > p.U1 - 1) continue;
    if (t >= Tb || u > Ub) continue;
    const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;

    // token logits [0, V): running max / sum of exp per lane
    float m = -INFINITY, s = 0.0f;
    for (long long k0 = 0; k0 < p.V; k0 += 32 * kUnroll) {
      float x[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const long long k = k0 + j * 32 + lane;
        x[j] = (k < p.V) ? Elem<DT>::load(row + k) : -INFINITY;
      }
      float cm = x[0];
#pragma unroll
      for (int j = 1; j < kUnroll; ++j) cm = fmaxf(cm, x[j]);
      if (cm > m) {
        s *= fast_exp2((m - cm) * kLog2e);
        m = cm;
      }
      if (m != -INFINITY) {
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) s += fast_exp2((x[j] - m) * kLog2e);
      }
    }
    const float M = warp_max(m);
    const float S = warp_sum(m == -INFINITY ? 0.0f : s * fast_exp2((m - M) * kLog2e));
    const fx_t lse_fx = fx_from_float(M) + fx_log_ge1(S);

    // duration logits [V, V+D): one lane per duration
    const float zd = (lane < p.D) ? Elem<DT>::load(row + p.V + lane) : -INFINITY;
    const float Md = warp_max(zd);
    const float Sd = warp_sum(lane < p.D ? fast_exp2((zd - Md) * kLog2e) : 0.0f);
    const fx_t lsed_fx = fx_from_float(Md) + fx_log_ge1(Sd);

    const long long q = diag_index(p, b, t, u);
    if (lane < p.D) ws.lpd[(long long)lane * ndiag_total + q] = clamp_lp(fx_from_float(zd) - lsed_fx);
    if (lane == 0) {
      const float zb = Elem<DT>::load(row + p.blank);
      ws.wb[q] = clamp_lp(fx_from_float(zb) - lse_fx) - p.sigma_fx;
      fx_t wl = kFxNegInf;
      if (u < Ub) {
        const long long y = p.labels[b * (p.U1 - 1) + u];
        if (y >= 0 && y < p.V && y != p.blank)
          wl = clamp_lp(fx_from_float(Elem<DT>::load(row + y)) - lse_fx) - p.sigma_fx;
      }
      ws.wl[q] = wl;
      ws.lse_tok[n] = M + logf(S);
      ws.lse_dur[n] = Md + logf(Sd);
    }
  }
}

}  // namespace

cudaError_t launch_node_tables(const Problem &p, int dtype, const Workspace &ws,
                               cudaStream_t stream) {
  const long long nodes = p.B * p.T * p.U1;
  if (nodes == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long warps_per_block = kTablesThreads / 32;
  long long blocks = (nodes + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  dim3 grid((unsigned)blocks), block(kTablesThreads);
  switch (dtype) {
    case kF32: node_tables_kernel<kF32><<<grid, block, 0, stream>>>(p, ws); break;
    case kF16: node_tables_kernel<kF16><<<grid, block, 0, stream>>>(p, ws); break;
    default: node_tables_kernel<kBF16><<<grid, block, 0, stream>>>(p, ws); break;
  }
  return cudaGetLastError();
}

}  // namespace tdt
