// tdt_tables.cu -- K1: per-node log-softmax tables.
//
// "log-softmax over the vocabulary for each lattice node" ("tdt-loss: add
// TDT loss kernel", kernels-community PR #882, "What's in it"), plus the
// log-softmax of the duration logits.  A group of TPR threads streams one
// logits row z[b,t,u,0:V+D) once: a scalar head up to the first 16-byte
// boundary, a body of 16-byte loads (each thread issues kBatch independent
// loads before touching any, so many bytes are in flight per SM), a scalar
// tail (tdt_rowio.cuh).  Each thread keeps a running max and a running sum
// of exp(z - max) in fp32; the group combines them with shuffles ("Warp
// Shuffle Reductions", "cuda-kernels" skill page) and, for groups wider than
// a warp, through shared memory.  TPR grows with the row length (4 threads
// for fp32 rows of up to 256 floats, 8 for 16-bit rows of up to 1024, a
// warp from ~2000 floats up), so the per-row work is amortised over many
// vectors per thread.
// The row may be a slice of a wider tensor: only strides s0..s2 locate it.
//
// Outputs per usable node (t < T_b, u <= U_b):
//   lse_tok[n], lse_dur[n]   float, for the gradient pass
//   arcw[g][0..2D)           node arc record of xf values (tdt_common.cuh):
//                            blank and label arc probabilities per duration,
//                            anti-diagonal layout, one contiguous record per
//                            node for the lattice passes
// and usable[b] = 1, ticket[b] = 0 for every utterance of the launch; with
// Problem::gx_rows > 0 also the alpha / beta entries of the band boundary
// rows set to lv_unwritten().
#include <type_traits>

#include "tdt_rowio.cuh"

namespace tdt {

namespace {

constexpr int kTablesThreads = 256;
constexpr int kBatch = 8;          // 16-byte loads issued per thread before use
constexpr int kVecPerThread = 16;  // row vectors per thread when choosing TPR


// (b, t, u) of row slot k when each utterance's T * U1 rows are walked
// u-major: k = (b * U1 + u) * T + t; 32-bit divisions as above.
__device__ __forceinline__ void decode_slot_umajor(const Problem &p, long long k, long long *b,
                                                   long long *t, long long *u) {
  const unsigned kk = (unsigned)k, U1 = (unsigned)p.U1, T = (unsigned)p.T;
  const unsigned bu = fast_div(kk, p.divT_m, p.divT_s);
  *t = kk - bu * T;
  const unsigned bb = fast_div(bu, p.divU1_m, p.divU1_s);
  *u = bu - bb * U1;
  *b = bb;
}

__device__ __forceinline__ fx_t clamp_lp(fx_t v) {
  const fx_t floor_fx = (fx_t)kLogProbFloor * (fx_t)4294967296LL;
  return v < floor_fx ? floor_fx : v;
}

// Merge two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void merge_ms(float &m, float &s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * fast_exp2((m - M) * kLog2e) + s2 * fast_exp2((m2 - M) * kLog2e);
  m = M;
}

// Combine (m, s) over the TPR threads of each row group of the block.
// Every thread of the block must call it (it may use __syncthreads).
template <int TPR>
__device__ __forceinline__ void group_ms(float &m, float &s, float *sm_m, float *sm_s) {
  constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
  for (int o = 1; o < W; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, m2, s2);
  }
  if constexpr (TPR > 32) {
    constexpr int NW = TPR / 32;  // warps per group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
      sm_m[warp] = m;
      sm_s[warp] = s;
    }
    __syncthreads();
    const int g0 = (warp / NW) * NW;
    m = sm_m[g0];
    s = sm_s[g0];
#pragma unroll
    for (int w = 1; w < NW; ++w) merge_ms(m, s, sm_m[g0 + w], sm_s[g0 + w]);
    __syncthreads();
  }
}

// Per-row values computed once per row group instead of by every lane:
// lane 0 of the group takes the token side, lane 1 the duration side, lanes 2
// and 3 the blank and label logits, and each of the four converts its value(s)
// to fx in the same two 64-bit conversions (which run on the slow float64
// pipe); the results are broadcast with shuffles.  Every lane of the warp
// calls it (inactive rows with neutral inputs), TPR >= 4.
struct RowScalars {
  fx_t lse_fx, lsed_fx;  // token and duration log-sum-exps in fx
  fx_t zb_fx, zy_fx;     // blank and label logits in fx
  float lse, lsed;       // the same log-sum-exps in fp32 (lane 0 / lane 1)
};

template <int TPR>
__device__ __forceinline__ RowScalars row_scalars(int lt, float M, float S, float md, float sd,
                                                  float zb, float zy, bool has_dur) {
  // ln(ss) = e ln2 + log1p(f - 1), ss = f 2^e, f in [1, 2): ss >= 1 (the
  // largest term of a sum taken relative to its maximum is 1)
  float mm = 0.0f, ss = 1.0f;
  if (lt == 0) { mm = M; ss = S; }
  if (lt == 1 && has_dur) { mm = md; ss = sd; }
  if (!(ss >= 1.0f) || !(mm > -INFINITY)) { mm = 0.0f; ss = 1.0f; }  // inactive rows
  const int bits = __float_as_int(ss);
  const int e = ((bits >> 23) & 0xff) - 127;
  const float f = __int_as_float((bits & 0x007fffff) | 0x3f800000);
  const float lf = log1pf(f - 1.0f);
  // the two conversions: lanes 0, 1: (lf, mm); lane 2: zb; lane 3: zy
  const float a = lt < 2 ? lf : (lt == 2 ? zb : zy);
  const fx_t v = fx_from_float(a) + (lt < 2 ? fx_from_float(mm) + (fx_t)e * kFxLn2 : (fx_t)0);
  constexpr int W = TPR < 32 ? TPR : 32;
  const int base = (threadIdx.x & 31) & ~(W - 1);
  RowScalars r;
  r.lse_fx = __shfl_sync(0xffffffffu, v, base);
  r.lsed_fx = __shfl_sync(0xffffffffu, v, base + 1);
  r.zb_fx = __shfl_sync(0xffffffffu, v, base + 2);
  r.zy_fx = __shfl_sync(0xffffffffu, v, base + 3);
  r.lse = r.lsed = mm + ((float)e * 0.6931471805599453f + lf);
  return r;
}

// Outputs of one usable node from its reduced row: the two log-sum-exps
// and the arc record -- [i] blank arc with duration i, [n_dur + i] label arc
// with duration i, each the arc's probability exp(token log-prob - sigma +
// duration log-prob) as an xf value, the log-weight summed in fx first.
// Lane lt of the row group holds durations lt, lt + TPR, ... in zd.
template <int TPR, int DPL>
__device__ __forceinline__ void write_node_outputs(const Problem &p, const Workspace &ws,
                                                   long long n, long long b, long long t,
                                                   long long u, int lt, const RowScalars &rs,
                                                   const float *zd, bool y_ok) {
  const fx_t wbs = clamp_lp(rs.zb_fx - rs.lse_fx) - p.sigma_fx;
  const fx_t wls = y_ok ? clamp_lp(rs.zy_fx - rs.lse_fx) - p.sigma_fx : 0;
  LV *rec = ws.arcw + diag_index(p, b, t, u) * p.rec_len;
  if (p.rnnt) {
    // plain RNN-T: no duration head; the blank arc advances one frame, the
    // label arc none; the other arcs of the lattice's {0, 1} get probability 0
    if (lt < p.n_dur) {
      rec[lt] = p.dur[lt] == 1 ? xf_from_fx(wbs) : xf_zero();
      rec[p.n_dur + lt] = p.dur[lt] == 0 ? xf_from_fx(wls) : xf_zero();
    }
  } else {
#pragma unroll
    for (int c = 0; c < DPL; ++c) {
      const int i = lt + c * TPR;
      if (i < p.D) {
        const fx_t ld = clamp_lp(fx_from_float(zd[c]) - rs.lsed_fx);
        rec[i] = xf_from_fx(wbs + ld);
        rec[p.n_dur + i] = xf_from_fx(wls + ld);
      }
    }
  }
  if (lt == 0) ws.lse_tok[n] = rs.lse;
  if (lt == 1) ws.lse_dur[n] = p.D > 0 ? rs.lsed : 0.0f;
  if (p.gx_rows > 0 && lt == 0) {
    // the rows that the lattice bands of this launch hand to a neighbour
    // through global memory (the top row of every band but the last for
    // alpha, the bottom row of every band but the first for beta) start
    // unwritten: the neighbour polls them until they are not
    const long long g = diag_index(p, b, t, u);
    const int m = (int)u % p.gx_rows;
    if (m == p.gx_rows - 1 && u + 1 < p.U1) ws.alpha[g] = lv_unwritten();
    if (m == 0 && u > 0) ws.beta[g] = lv_unwritten();
  }
}

// Largest element of a batch of 16-byte vectors (those with index < nvec):
// 16-bit types by packed pairwise maxima (one instruction per two elements)
// before converting, fp32 element by element.
template <int DT, int KB, int TPR>
__device__ __forceinline__ float batch_max(const uint4 *v, int j0, int lt, int nvec) {
  if constexpr (DT == kF32) {
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      if (j0 + i * TPR + lt < nvec) {
        cm = fmaxf(cm, fmaxf(fmaxf(__uint_as_float(v[i].x), __uint_as_float(v[i].y)),
                             fmaxf(__uint_as_float(v[i].z), __uint_as_float(v[i].w))));
      }
    }
    return cm;
  } else {
    typedef typename std::conditional<DT == kBF16, __nv_bfloat162, __half2>::type H2;
    const unsigned neg_inf_pair = DT == kBF16 ? 0xff80ff80u : 0xfc00fc00u;
    unsigned acc = neg_inf_pair;
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      if (j0 + i * TPR + lt < nvec) {
        const unsigned w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          H2 a = *reinterpret_cast<const H2 *>(&acc), bb = *reinterpret_cast<const H2 *>(&w[k]);
          H2 r = __hmax2(a, bb);
          acc = *reinterpret_cast<const unsigned *>(&r);
        }
      }
    }
    float x[2];
    if constexpr (DT == kBF16) {
      x[0] = __uint_as_float(acc << 16);
      x[1] = __uint_as_float(acc & 0xffff0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&acc));
      x[0] = f.x;
      x[1] = f.y;
    }
    return fmaxf(x[0], x[1]);
  }
}

template <int DT, int TPR, int DPL>
__global__ void __launch_bounds__(kTablesThreads, 4)
node_tables_kernel(Problem p, Workspace ws, long long n_begin, long long n_end) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  constexpr int RPB = kTablesThreads / TPR;
  constexpr int kDurPerLane = DPL;  // duration logits a lane holds (D <= TPR * DPL)
  __shared__ float sm_m[kTablesThreads / 32], sm_s[kTablesThreads / 32];
  const E *logits = static_cast<const E *>(p.logits);
  const int lt = threadIdx.x % TPR;
  // A launch covers whole utterances: mark them usable before their lattice
  // passes run (those clear the flag of an utterance with unusable lengths or
  // labels, or whose bounded wait gave up).
  if (blockIdx.x == 0) {
    const long long per_utt = p.T * p.U1;
    for (long long bb = n_begin / per_utt + threadIdx.x; bb < n_end / per_utt; bb += blockDim.x) {
      ws.usable[bb] = 1;
      ws.ticket[bb] = 0;
    }
  }
  // The row slots of a launch walk each utterance u-major (t fastest), so
  // the RPB rows of a block share u and, with ragged label lengths, a block
  // is either all padding (u > U_b, it ends at once) or all lattice rows
  // instead of a few active rows among padding ones (measured: bf16 sliced
  // workload 0.360 vs 0.367 ms, large_batch 1.903 vs 1.914 ms, parakeet
  // unchanged).  A launch covers whole utterances.
  const long long slot = n_begin + (long long)blockIdx.x * RPB + threadIdx.x / TPR;
  long long b = 0, t = 0, u = 0, Ub = 0, n = 0;
  bool active = slot < n_end;
  if (active) {
    decode_slot_umajor(p, slot, &b, &t, &u);
    n = (b * p.T + t) * p.U1 + u;
    const long long Tb = p.logit_lens[b];
    Ub = p.label_lens[b];
    active = Tb >= 1 && Tb <= p.T && Ub >= 0 && Ub <= p.U1 - 1 && t < Tb && u <= Ub;
  }
  const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;

  // Everything of the row that does not depend on its reduction is loaded up
  // front, so the row costs one memory round trip (plus one for the label's
  // logit) rather than one per part: the duration logits (lane lt holds
  // durations lt, lt + TPR, ...), the blank logit, the label and its logit.
  float zd[kDurPerLane];
  float zb = 0.0f, zy = 0.0f;
  long long y = -1;
  int head = 0, nvec = 0, ntail = 0;
  float zh = 0.0f, zt = 0.0f;
  if (active) {
#pragma unroll
    for (int c = 0; c < kDurPerLane; ++c) {
      const int i = lt + c * TPR;
      zd[c] = i < p.D ? Elem<DT>::load(row + p.V + i) : -INFINITY;
    }
    zb = Elem<DT>::load(row + p.blank);
    if (u < Ub) y = p.labels[b * (p.U1 - 1) + u];
    head = head_elems<DT>(row);
    if (head > p.V) head = (int)p.V;
    nvec = (int)((p.V - head) / N);
    const int tail0 = head + nvec * N;
    ntail = (int)(p.V - tail0);
    // head (< N elements) and tail (< N elements) each on lanes 0.., TPR >= N
    if (lt < head) zh = Elem<DT>::load(row + lt);
    if (lt < ntail) zt = Elem<DT>::load(row + tail0 + lt);
  }
  const bool y_ok = y >= 0 && y < p.V && y != p.blank;

  // token logits [0, V)
  float m = -INFINITY, s = 0.0f, mL = -INFINITY;
  if (active) {
    const uint4 *vbase = reinterpret_cast<const uint4 *>(row + head);
    for (int j0 = 0; j0 < nvec; j0 += TPR * kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i * TPR + lt;
        if (j < nvec) v[i] = ld_row16<false>(vbase + j);
      }
      // the label's logit, once the label has arrived (overlaps the batch)
      if (j0 == 0 && y_ok) zy = Elem<DT>::load(row + y);
      const float cm = batch_max<DT, kBatch, TPR>(v, j0, lt, nvec);
      if (cm > m) {
        s *= fast_exp2((m - cm) * kLog2e);
        m = cm;
        mL = m * kLog2e;
      }
      if (m != -INFINITY) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (j0 + i * TPR + lt < nvec) {
            float x[N];
            unpack<DT>(v[i], x);
            // x log2(e) - m log2(e) in one rounding; the rounding of m log2(e)
            // is common to the row's terms (a relative 2^-24 of m log2 e)
#pragma unroll
            for (int e = 0; e < N; ++e) s += fast_exp2(fmaf(x[e], kLog2e, -mL));
          }
        }
      }
    }
    if (nvec == 0 && y_ok) zy = Elem<DT>::load(row + y);
    if (lt < head) merge_ms(m, s, zh, 1.0f);
    if (lt < ntail) merge_ms(m, s, zt, 1.0f);
  }
  group_ms<TPR>(m, s, sm_m, sm_s);
  const float M = m, S = s;

  // duration logits [V, V+D)
  float md = -INFINITY, sd = 0.0f;
  if (active) {
#pragma unroll
    for (int c = 0; c < kDurPerLane; ++c)
      if (lt + c * TPR < p.D) merge_ms(md, sd, zd[c], 1.0f);
  }
  group_ms<TPR>(md, sd, sm_m, sm_s);
  const RowScalars rs = row_scalars<TPR>(lt, M, S, md, sd, zb, zy, p.D > 0);
  if (!active) return;
  write_node_outputs<TPR, kDurPerLane>(p, ws, n, b, t, u, lt, rs, zd, y_ok);
}

template <int DT, int TPR, int DPL>
cudaError_t launch_tpr_dpl(const Problem &p, const Workspace &ws, long long n_begin,
                           long long n_end, cudaStream_t stream) {
  constexpr int RPB = kTablesThreads / TPR;
  const long long rows = n_end - n_begin;
  const long long blocks = (rows + RPB - 1) / RPB;
  node_tables_kernel<DT, TPR, DPL>
      <<<(unsigned)blocks, kTablesThreads, kStreamSmemReserve, stream>>>(p, ws, n_begin, n_end);
  return cudaGetLastError();
}

// Duration logits per lane: the fewest (1, 2 or 4, else all that D may
// need) that hold the problem's D.
template <int DT, int TPR>
cudaError_t launch_tpr(const Problem &p, const Workspace &ws, long long n_begin, long long n_end,
                       cudaStream_t stream) {
  constexpr int kFull = (kMaxDurations + TPR - 1) / TPR;
  const long long need = (p.D + TPR - 1) / TPR;
  if (need <= 1) return launch_tpr_dpl<DT, TPR, 1>(p, ws, n_begin, n_end, stream);
  if constexpr (kFull >= 2)
    if (need <= 2) return launch_tpr_dpl<DT, TPR, 2>(p, ws, n_begin, n_end, stream);
  if constexpr (kFull >= 4)
    if (need <= 4) return launch_tpr_dpl<DT, TPR, 4>(p, ws, n_begin, n_end, stream);
  return launch_tpr_dpl<DT, TPR, kFull>(p, ws, n_begin, n_end, stream);
}

template <int DT>
cudaError_t launch_dt(const Problem &p, const Workspace &ws, long long n_begin, long long n_end,
                      cudaStream_t stream) {
  // a warp per long row (no shared-memory combine), fewer lanes for short rows
  const long long row_bytes = p.V * (long long)sizeof(typename Elem<DT>::T);
  int tpr = row_group_threads(row_bytes, kVecPerThread);
  if (tpr > 32) tpr = 32;
  // fp32 rows of up to 1 KB: 4 lanes (one 4-element vector of scalar head or
  // tail per lane), so a warp's per-row work (the group combines, the
  // duration softmax, the record) serves 8 rows instead of 4
  if constexpr (Vec<DT>::N <= 4) {
    if (row_bytes <= 4 * kVecPerThread * 16)
      return launch_tpr<DT, 4>(p, ws, n_begin, n_end, stream);
  }
  switch (tpr) {
    case 8: return launch_tpr<DT, 8>(p, ws, n_begin, n_end, stream);
    case 16: return launch_tpr<DT, 16>(p, ws, n_begin, n_end, stream);
    case 32: return launch_tpr<DT, 32>(p, ws, n_begin, n_end, stream);
    case 64: return launch_tpr<DT, 64>(p, ws, n_begin, n_end, stream);
    case 128: return launch_tpr<DT, 128>(p, ws, n_begin, n_end, stream);
    default: return launch_tpr<DT, 256>(p, ws, n_begin, n_end, stream);
  }
}

}  // namespace

cudaError_t launch_node_tables(const Problem &p, int dtype, const Workspace &ws,
                               long long n_begin, long long n_end, cudaStream_t stream) {
  if (n_end - n_begin <= 0) return cudaSuccess;
  switch (dtype) {
    case kF32: return launch_dt<kF32>(p, ws, n_begin, n_end, stream);
    case kF16: return launch_dt<kF16>(p, ws, n_begin, n_end, stream);
    default: return launch_dt<kBF16>(p, ws, n_begin, n_end, stream);
  }
}

}  // namespace tdt
