// tdt_tables.cu -- K1: per-node log-softmax tables.
//
// "log-softmax over the vocabulary for each lattice node" ("tdt-loss: add
// TDT loss kernel", kernels-community PR #882, "What's in it"), plus the
// log-softmax of the duration logits.  One warp streams one logits row
// z[b,t,u,0:V+D) once with 16-byte loads (scalar head/tail, see
// tdt_rowio.cuh), keeping a running max and a running sum of exp(z - max)
// per lane in fp32, then combines lanes with shuffles ("Warp Shuffle
// Reductions", "cuda-kernels" skill page).  The row may be a slice of a
// wider tensor: only strides s0..s2 locate it.  One warp per row and no grid
// stride, so the blocks are short and other kernels can be scheduled
// between them.
//
// Outputs per usable node (t < T_b, u <= U_b):
//   lse_tok[n], lse_dur[n]   float, for the gradient pass
//   arcw[g][0..2D)           fx arc log-weights lpB - sigma + lpD_i and
//                            lpL - sigma + lpD_i, anti-diagonal layout, one
//                            contiguous record per node for the lattice passes
#include "tdt_rowio.cuh"

namespace tdt {

namespace {

constexpr int kTablesThreads = 256;
constexpr int kTablesUnroll = 4;  // 16-byte vectors in flight per lane per iteration

__device__ __forceinline__ fx_t clamp_lp(fx_t v) {
  const fx_t floor_fx = (fx_t)kLogProbFloor * (fx_t)4294967296LL;
  return v < floor_fx ? floor_fx : v;
}

template <int DT>
__global__ void __launch_bounds__(kTablesThreads)
node_tables_kernel(Problem p, Workspace ws, long long n_begin, long long n_end) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  const E *logits = static_cast<const E *>(p.logits);
  const int lane = threadIdx.x & 31;
  const long long n = n_begin + (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (n >= n_end) return;
  const long long u = n % p.U1;
  const long long bt = n / p.U1;
  const long long t = bt % p.T;
  const long long b = bt / p.T;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  if (Tb < 1 || Tb > p.T || Ub < 0 || Ub > p.U1 - 1) return;
  if (t >= Tb || u > Ub) return;
  const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;

  // token logits [0, V): scalar head and tail first, then 16-byte vectors
  int head = head_elems<DT>(row);
  if (head > p.V) head = (int)p.V;
  const long long nvec = (p.V - head) / N;
  const long long tail0 = head + nvec * N;
  const int ntail = (int)(p.V - tail0);
  float m = -INFINITY, s = 0.0f;
  if (lane < head) {
    m = Elem<DT>::load(row + lane);
    s = 1.0f;
  } else if (lane < head + ntail) {
    m = Elem<DT>::load(row + tail0 + (lane - head));
    s = 1.0f;
  }
  // Two batches of kTablesUnroll 16-byte vectors per lane: the next batch is
  // loaded before the math of the current one, so loads stay in flight.
  const uint4 *vbase = reinterpret_cast<const uint4 *>(row + head);
  const int nv = (int)nvec;
  uint4 cur[kTablesUnroll], nxt[kTablesUnroll];
#pragma unroll
  for (int k = 0; k < kTablesUnroll; ++k) {
    const int j = k * 32 + lane;
    if (j < nv) cur[k] = __ldg(vbase + j);
  }
  for (int j0 = 0; j0 < nv; j0 += 32 * kTablesUnroll) {
    const int jn = j0 + 32 * kTablesUnroll;
#pragma unroll
    for (int k = 0; k < kTablesUnroll; ++k) {
      const int j = jn + k * 32 + lane;
      if (j < nv) nxt[k] = __ldg(vbase + j);
    }
    float x[kTablesUnroll * N];
#pragma unroll
    for (int k = 0; k < kTablesUnroll; ++k) {
      if (j0 + k * 32 + lane < nv) {
        unpack<DT>(cur[k], x + k * N);
      } else {
#pragma unroll
        for (int e = 0; e < N; ++e) x[k * N + e] = -INFINITY;
      }
    }
    float cm = x[0];
#pragma unroll
    for (int e = 1; e < kTablesUnroll * N; ++e) cm = fmaxf(cm, x[e]);
    if (cm > m) {
      s *= fast_exp2((m - cm) * kLog2e);
      m = cm;
    }
    if (m != -INFINITY) {
      // (x - m) first: exact for the terms near the max, which dominate the sum
#pragma unroll
      for (int e = 0; e < kTablesUnroll * N; ++e) s += fast_exp2((x[e] - m) * kLog2e);
    }
#pragma unroll
    for (int k = 0; k < kTablesUnroll; ++k) cur[k] = nxt[k];
  }
  const float M = warp_max(m);
  const float S = warp_sum(m == -INFINITY ? 0.0f : s * fast_exp2((m - M) * kLog2e));
  const fx_t lse_fx = fx_from_float(M) + fx_log_ge1(S);

  // duration logits [V, V+D): one lane per duration
  const float zd = (lane < p.D) ? Elem<DT>::load(row + p.V + lane) : -INFINITY;
  const float Md = warp_max(zd);
  const float Sd = warp_sum(lane < p.D ? fast_exp2((zd - Md) * kLog2e) : 0.0f);
  const fx_t lsed_fx = fx_from_float(Md) + fx_log_ge1(Sd);

  // arc log-weights of this node: [i] blank arc with duration i, [D + i]
  // label arc with duration i (lane i writes both)
  fx_t wbs = 0, wls = 0;
  if (lane == 0) {
    const float zb = Elem<DT>::load(row + p.blank);
    wbs = clamp_lp(fx_from_float(zb) - lse_fx) - p.sigma_fx;
    if (u < Ub) {
      const long long y = p.labels[b * (p.U1 - 1) + u];
      if (y >= 0 && y < p.V && y != p.blank)
        wls = clamp_lp(fx_from_float(Elem<DT>::load(row + y)) - lse_fx) - p.sigma_fx;
    }
    ws.lse_tok[n] = M + logf(S);
    ws.lse_dur[n] = Md + logf(Sd);
  }
  wbs = __shfl_sync(0xffffffffu, wbs, 0);
  wls = __shfl_sync(0xffffffffu, wls, 0);
  if (lane < p.D) {
    const fx_t ld = clamp_lp(fx_from_float(zd) - lsed_fx);
    fx_t *rec = ws.arcw + diag_index(p, b, t, u) * (2 * p.D);
    rec[lane] = wbs + ld;
    rec[p.D + lane] = wls + ld;
  }
}

}  // namespace

cudaError_t launch_node_tables(const Problem &p, int dtype, const Workspace &ws,
                               long long n_begin, long long n_end, cudaStream_t stream) {
  const long long rows = n_end - n_begin;
  if (rows <= 0) return cudaSuccess;
  const long long warps_per_block = kTablesThreads / 32;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  dim3 grid((unsigned)blocks), block(kTablesThreads);
  switch (dtype) {
    case kF32: node_tables_kernel<kF32><<<grid, block, 0, stream>>>(p, ws, n_begin, n_end); break;
    case kF16: node_tables_kernel<kF16><<<grid, block, 0, stream>>>(p, ws, n_begin, n_end); break;
    default: node_tables_kernel<kBF16><<<grid, block, 0, stream>>>(p, ws, n_begin, n_end); break;
  }
  return cudaGetLastError();
}

}  // namespace tdt
