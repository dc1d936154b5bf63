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
// A group of TPR threads takes one row (a whole block for rows of 16 KB or
// more): each thread issues kBatch independent 16-byte loads, then computes
// and stores them as 16-byte vectors, when the input row and the output row
// sit at the same offset from a 16-byte boundary (the contiguous case);
// otherwise (a strided view) it stores output-aligned 16-byte vectors, each
// assembled from the two aligned input vectors it spans.  The row's
// coefficients (N, fB, fL, fD_i, the saved log-sum-exps, the label) are read
// from the lattice pass's outputs together with the row's first batch of
// logits, so their latencies overlap; every lane of a row group computes
// them (the loads are broadcasts within a warp).
#include "tdt_async.cuh"
#include "tdt_rowio.cuh"

namespace tdt {

extern __shared__ __align__(16) unsigned char tdt_dyn_smem[];

namespace {

constexpr int kGradThreads = 256;
constexpr int kVecPerThread = 8;      // row vectors per lane when choosing TPR
constexpr int kLongRowBytes = 16384;  // rows from this size on: one block per row
constexpr int kStagedViewTPR = 64;    // lanes per realigned long row (staged)

// 16-byte chunks of one row's staging buffer: the row's token logits plus
// one chunk at each end for the misalignment.
__host__ __device__ inline int stage_chunks(long long v_bytes) { return (int)(v_bytes / 16) + 2; }

// 16-byte loads a lane issues before it uses them, and the blocks per SM the
// registers are sized for.  Measured on GB300: 8 loads for one block per row
// (a long row in one batch) and for 8-lane groups; 4 loads otherwise, which
// keeps the kernel within 64 registers (four blocks per SM) without spills.
template <int TPR> struct GradShape {
  static constexpr int kBatch = (TPR == 256 || TPR == 8) ? 8 : 4;
  static constexpr int kMinBlocks = TPR == 8 ? 3 : 4;
};

template <int DT, int TPR>
__device__ __forceinline__ void zero_row(typename Elem<DT>::T *out, long long VD, int lt) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  int head = head_elems<DT>(out);
  if (head > VD) head = (int)VD;
  const int nvec = (int)((VD - head) / N);
  const long long tail0 = head + (long long)nvec * N;
  const E zero = Elem<DT>::from_float(0.0f);
  if (lt < head) out[lt] = zero;
  if (lt < VD - tail0) out[tail0 + lt] = zero;
  uint4 *v = reinterpret_cast<uint4 *>(out + head);
  for (int j = lt; j < nvec; j += TPR) v[j] = make_uint4(0u, 0u, 0u, 0u);
}

// VIEW: the logits rows may sit at another offset from a 16-byte boundary
// than the gradient rows (a strided view); without it every row is known to
// share the gradient row's alignment (one contiguous layout).  STAGE: the
// row's 16-byte chunks go to shared memory by cp.async (see below) instead
// of being loaded into registers in batches.
template <int DT, int TPR, bool COH, bool VIEW, bool STAGE>
__global__ void __launch_bounds__(kGradThreads, GradShape<TPR>::kMinBlocks)
grad_kernel(Problem p, Workspace ws, typename Elem<DT>::T *grad, const float *gscale,
            long long n_begin, long long n_end) {
  typedef typename Elem<DT>::T E;
  constexpr int N = Vec<DT>::N;
  constexpr int RPB = kGradThreads / TPR;
  constexpr int kBatch = GradShape<TPR>::kBatch;
  constexpr int kDurPerLane = (kMaxDurations + TPR - 1) / TPR;  // D <= kMaxDurations
  const E *logits = static_cast<const E *>(p.logits);
  const int lt = threadIdx.x % TPR;
  const long long n = n_begin + (long long)blockIdx.x * RPB + threadIdx.x / TPR;
  if (n >= n_end) return;
  long long b, t, u;
  decode_node(p, n, &b, &t, &u);
  E *out = grad + n * p.VD;
  const long long Tb = p.logit_lens[b], Ub = p.label_lens[b];
  const E *row = logits + b * p.s0 + t * p.s1 + u * p.s2;
  const bool in_lattice = t < Tb && u <= Ub;
  // Everything the row needs is loaded up front, so its latencies overlap:
  // the first batch of 16-byte vectors, the scalar head and tail, the
  // duration logits and their fractions (lane lt: durations lt, lt + TPR,
  // ...), alpha, beta and the other lattice outputs of the row, and the
  // upstream gradient.
  const uintptr_t ai = reinterpret_cast<uintptr_t>(row), ao = reinterpret_cast<uintptr_t>(out);
  // without VIEW the host has checked that every row shares the output's alignment
  const bool vec = !VIEW || ((ai ^ ao) & 15) == 0;
  int head = head_elems<DT>(row);
  if (head > p.V) head = (int)p.V;
  const int nvec = (int)((p.V - head) / N);
  const long long tail0 = head + (long long)nvec * N;
  const int ntail = (int)(p.V - tail0);
  const uint4 *vin = reinterpret_cast<const uint4 *>(row + head);
  uint4 v[kBatch];
  float zh = 0.0f, zt = 0.0f, zd[kDurPerLane], fd[kDurPerLane];
  LV al = {}, be = {}, ll = {};
  float sc = 0.0f;
  int usable = 0;
  float lse_t = 0.0f, lse_d = 0.0f, fb = 0.0f, fl = 0.0f;
  long long y = -1;
  // Staged rows: the aligned 16-byte chunks of the row that lie wholly
  // inside its token logits go to the row group's shared buffer by cp.async
  // before anything else, so no register is held while they are in flight.
  // A row at the gradient row's 16-byte offset takes chunk j for output
  // vector j, each lane reading back only the chunks it copied.  A realigned
  // row (a strided view at another offset) takes for output vector j (the
  // 16 bytes at `first` + 16 j of the input) chunk j funnel-shifted with
  // chunk j + 1, copied by the next lane.
  // (a strided view stages only its realigned rows: the few rows that meet
  // the gradient's offset keep the register batches)
  constexpr bool kStaged = STAGE;
  constexpr bool kStagedAligned = STAGE && !VIEW;
  int oh = 0, onv = 0, sh = 0, c_lo = 0, c_hi = 0;
  uintptr_t abase = 0;
  uint4 *stage = nullptr;
  if constexpr (kStaged) {
    stage = reinterpret_cast<uint4 *>(tdt_dyn_smem) +
            (threadIdx.x / TPR) * stage_chunks((long long)p.V * sizeof(E));
    if (kStagedAligned && in_lattice && vec) {
      for (int c = lt; c < nvec; c += TPR) cp_async16(stage + c, vin + c);
      cp_async_commit();
    } else if (VIEW && in_lattice && !vec) {
      oh = head_elems<DT>(out);
      if (oh > p.V) oh = (int)p.V;
      onv = (int)((p.V - oh) / N);
      const uintptr_t rlo = ai, rhi = ai + (uintptr_t)p.V * sizeof(E);
      const uintptr_t first = ai + (uintptr_t)oh * sizeof(E);
      sh = (int)(first & 15);
      abase = first - (uintptr_t)sh;
      c_lo = abase >= rlo ? 0 : 1;
      c_hi = (int)((rhi - abase) / 16);
      if (c_hi > onv + 1) c_hi = onv + 1;
      for (int c = c_lo + lt; c < c_hi; c += TPR)
        cp_async16(stage + c, reinterpret_cast<const void *>(abase + 16 * (uintptr_t)c));
      cp_async_commit();
    }
  }
  if (in_lattice) {
    if (vec) {
      if constexpr (!kStagedAligned) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int j = i * TPR + lt;
          if (j < nvec) v[i] = ld_row16<COH>(vin + j);
        }
      }
      if (lt < head) zh = ld_elem<DT, COH>(row + lt);
      if (lt < ntail) zt = ld_elem<DT, COH>(row + tail0 + lt);
    }
    const long long q = diag_index(p, b, t, u);
    const float *fr = ws.frac + q * (2 + p.n_dur);  // the node's fraction record
#pragma unroll
    for (int c = 0; c < kDurPerLane; ++c) {
      const int i = lt + c * TPR;
      zd[c] = i < p.D ? ld_elem<DT, COH>(row + p.V + i) : 0.0f;
      fd[c] = i < p.D ? fr[2 + i] : 0.0f;
    }
    al = ws.alpha[q];
    be = ws.beta[q];
    ll = ws.loglik[b];
    sc = ws.scale[b];
    usable = ws.usable[b];
    lse_t = ws.lse_tok[n];
    lse_d = ws.lse_dur[n];
    fb = fr[0];
    fl = fr[1];
    if (u < Ub) y = p.labels[b * (p.U1 - 1) + u];
  }
  // upstream gradient of utterance b's loss (1 when none is given; x * 1 is exact)
  const float gs = gscale ? gscale[p.reduction == kNone ? b : 0] : 1.0f;
  // rows outside a usable lattice, or of zero occupancy, get a zero gradient
  if (!in_lattice || !usable || al.s == 0.0f || be.s == 0.0f || ll.s == 0.0f) {
    if constexpr (kStaged) cp_async_wait<0>();  // no copy outlives its thread
    zero_row<DT, TPR>(out, p.VD, lt);
    return;
  }
  // c_b N with the occupancy N = alpha beta / L = 2^k s_a s_b / s_L,
  // k = e_a + e_b - e_L (N <= 1, so k <= 2): 2^k as an exact fp32 power of two
  const int k2 = min(max(al.e + be.e - ll.e + 127, 0), 254);
  const float a0 = sc * (__int_as_float(k2 << 23) * (al.s * be.s / ll.s));
  const float a = a0 * gs, lse2 = lse_t * kLog2e, lsed2 = lse_d * kLog2e;
  const float ab = (a0 * fb) * gs, alb = (a0 * fl) * gs;
  auto g_at = [&](float x, long long k) {
    float g = a * fast_exp2(fmaf(x, kLog2e, -lse2));
    if (k == p.blank) g -= ab;
    if (k == y) g -= alb;
    return g;
  };

  if (vec) {
    if (lt < head) out[lt] = Elem<DT>::from_float(g_at(zh, lt));
    if (lt < ntail) out[tail0 + lt] = Elem<DT>::from_float(g_at(zt, tail0 + lt));
    uint4 *vout = reinterpret_cast<uint4 *>(out + head);
    // vectors holding the two special entries (or -1)
    const int jb = (p.blank >= head && p.blank < tail0) ? (int)((p.blank - head) / N) : -1;
    const int jy = (y >= head && y < tail0) ? (int)((y - head) / N) : -1;
    const int eb = (int)((p.blank - head) % N), ey = (int)((y - head) % N);
    if constexpr (kStagedAligned) {
      cp_async_wait<0>();  // the lane's own chunks, the only ones it reads
      for (int j = lt; j < nvec; j += TPR) {
        float x[N];
        unpack<DT>(stage[j], x);
        const int kb = j == jb ? eb : -1, ky = j == jy ? ey : -1;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          x[e] = a * fast_exp2(fmaf(x[e], kLog2e, -lse2));
          if (e == kb) x[e] -= ab;
          if (e == ky) x[e] -= alb;
        }
        vout[j] = pack<DT>(x);
      }
    } else {
    for (int j0 = 0; j0 < nvec; j0 += TPR * kBatch) {
      if (j0 > 0) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int j = j0 + i * TPR + lt;
          if (j < nvec) v[i] = ld_row16<COH>(vin + j);
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i * TPR + lt;
        if (j < nvec) {
          float x[N];
          unpack<DT>(v[i], x);
#pragma unroll
          for (int e = 0; e < N; ++e) x[e] = a * fast_exp2(fmaf(x[e], kLog2e, -lse2));
          if (j == jb) x[eb] -= ab;
          if (j == jy) x[ey] -= alb;
          vout[j] = pack<DT>(x);
        }
      }
    }
    }
  } else if constexpr (kStaged && VIEW) {
    const long long ot0 = oh + (long long)onv * N;
    if (lt < oh) out[lt] = Elem<DT>::from_float(g_at(ld_elem<DT, COH>(row + lt), lt));
    if (lt < p.V - ot0)
      out[ot0 + lt] = Elem<DT>::from_float(g_at(ld_elem<DT, COH>(row + ot0 + lt), ot0 + lt));
    uint4 *vout = reinterpret_cast<uint4 *>(out + oh);
    const int jb = (p.blank >= oh && p.blank < ot0) ? (int)((p.blank - oh) / N) : -1;
    const int jy = (y >= oh && y < ot0) ? (int)((y - oh) / N) : -1;
    const int eb = (int)((p.blank - oh) % N), ey = (int)((y - oh) % N);
    const int qw = sh >> 2, rb = (sh & 3) * 8;
    // every chunk of the row group has landed: own copies, then the group's
    // named barrier (ids 1, 2, ...: one per row group of the block)
    cp_async_wait<0>();
    if constexpr (TPR >= 32) {
      asm volatile("bar.sync %0, %1;" ::"r"(1 + (int)threadIdx.x / TPR), "r"(TPR) : "memory");
    } else {
      const unsigned lane = threadIdx.x & 31;
      __syncwarp(((1u << TPR) - 1u) << (lane & ~(unsigned)(TPR - 1)));
    }
    for (int j = lt; j < onv; j += TPR) {
      float x[N];
      if (j >= c_lo && j + (sh ? 1 : 0) < c_hi) {
        const uint4 lo = stage[j];
        unpack<DT>(sh ? funnel16(lo, stage[j + 1], qw, rb) : lo, x);
      } else {  // a vector whose input span leaves the row: element loads
        const long long k0 = oh + (long long)N * j;
#pragma unroll
        for (int e = 0; e < N; ++e) x[e] = ld_elem<DT, COH>(row + k0 + e);
      }
      // the blank and label entries by unrolled compares (a runtime index
      // into x would put it in local memory)
      const int kb = j == jb ? eb : -1, ky = j == jy ? ey : -1;
#pragma unroll
      for (int e = 0; e < N; ++e) {
        x[e] = a * fast_exp2(fmaf(x[e], kLog2e, -lse2));
        if (e == kb) x[e] -= ab;
        if (e == ky) x[e] -= alb;
      }
      vout[j] = pack<DT>(x);
    }
  } else if constexpr (VIEW) {
    // The input and output rows sit at different offsets from a 16-byte
    // boundary (a strided view of a wider tensor): output-aligned 16-byte
    // vectors, each assembled from the two aligned input vectors it spans
    // (the second is the next lane's first, served by L1).  Vectors whose
    // input span would leave the row, and the output's scalar head and
    // tail, take element accesses.
    int oh = head_elems<DT>(out);
    if (oh > p.V) oh = (int)p.V;
    const int onv = (int)((p.V - oh) / N);
    const long long ot0 = oh + (long long)onv * N;
    const uintptr_t rlo = reinterpret_cast<uintptr_t>(row);
    const uintptr_t rhi = rlo + (uintptr_t)p.V * sizeof(E);
    const uintptr_t first = reinterpret_cast<uintptr_t>(row + oh);
    const int sh = (int)(first & 15);  // the same for every output vector
    const int qw = sh >> 2, rb = (sh & 3) * 8;
    const uintptr_t abase = first - (uintptr_t)sh;
    if (lt < oh) out[lt] = Elem<DT>::from_float(g_at(ld_elem<DT, COH>(row + lt), lt));
    if (lt < p.V - ot0)
      out[ot0 + lt] = Elem<DT>::from_float(g_at(ld_elem<DT, COH>(row + ot0 + lt), ot0 + lt));
    uint4 *vout = reinterpret_cast<uint4 *>(out + oh);
    const int jb = (p.blank >= oh && p.blank < ot0) ? (int)((p.blank - oh) / N) : -1;
    const int jy = (y >= oh && y < ot0) ? (int)((y - oh) / N) : -1;
    const int eb = (int)((p.blank - oh) % N), ey = (int)((y - oh) % N);
    // One aligned input vector per output vector in flight: the 16 bytes
    // after it are the next lane's vector, taken by a shuffle; the last lane
    // of a warp's share of the row (and a lane whose neighbour has no vector)
    // loads them itself, in the same batch.
    constexpr int W = TPR < 32 ? TPR : 32;  // lanes of the row group within one warp
    const bool last_in_warp = (lt % W) == W - 1;
    constexpr int kFB = 4;
    for (int j0 = 0; j0 < onv; j0 += TPR * kFB) {
      uint4 lo[kFB], hi[kFB];
      bool lok[kFB], nok[kFB], hok[kFB];
#pragma unroll
      for (int i = 0; i < kFB; ++i) {
        const int j = j0 + i * TPR + lt;
        const uintptr_t A = abase + 16 * (uintptr_t)j;
        lok[i] = j < onv && A >= rlo && A + 16 <= rhi;
        // the neighbour lane's vector is the one at A + 16
        nok[i] = !last_in_warp && j + 1 < onv && A + 16 >= rlo && A + 32 <= rhi;
        hok[i] = nok[i];
        if (lok[i]) lo[i] = ld_row16<COH>(reinterpret_cast<const uint4 *>(A));
        if (sh && lok[i] && !nok[i] && A + 32 <= rhi) {
          hi[i] = ld_row16<COH>(reinterpret_cast<const uint4 *>(A + 16));
          hok[i] = true;
        }
      }
#pragma unroll
      for (int i = 0; i < kFB; ++i) {
        uint4 nb;
        nb.x = __shfl_down_sync(0xffffffffu, lo[i].x, 1);
        nb.y = __shfl_down_sync(0xffffffffu, lo[i].y, 1);
        nb.z = __shfl_down_sync(0xffffffffu, lo[i].z, 1);
        nb.w = __shfl_down_sync(0xffffffffu, lo[i].w, 1);
        if (nok[i]) hi[i] = nb;
        const int j = j0 + i * TPR + lt;
        if (j < onv) {
          const long long k0 = oh + (long long)N * j;
          float x[N];
          if (lok[i] && (sh == 0 || hok[i])) {
            unpack<DT>(funnel16(lo[i], sh ? hi[i] : lo[i], qw, rb), x);
          } else {
#pragma unroll
            for (int e = 0; e < N; ++e) x[e] = ld_elem<DT, COH>(row + k0 + e);
          }
#pragma unroll
          for (int e = 0; e < N; ++e) x[e] = a * fast_exp2(fmaf(x[e], kLog2e, -lse2));
          if (j == jb) x[eb] -= ab;
          if (j == jy) x[ey] -= alb;
          vout[j] = pack<DT>(x);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kDurPerLane; ++c) {
    const int i = lt + c * TPR;
    if (i < p.D)
      out[p.V + i] =
          Elem<DT>::from_float(a * fast_exp2(fmaf(zd[c], kLog2e, -lsed2)) - (a0 * fd[c]) * gs);
  }
}

template <int DT, int TPR>
cudaError_t launch_tpr(const Problem &p, const Workspace &ws, typename Elem<DT>::T *grad,
                       const float *gscale, long long n_begin, long long n_end,
                       cudaStream_t stream) {
  constexpr int RPB = kGradThreads / TPR;
  const long long rows = n_end - n_begin;
  const long long blocks = (rows + RPB - 1) / RPB;
  // the output overlaps the logits (written in place): coherent loads
  const char *lo = static_cast<const char *>(p.logits);
  const char *go = reinterpret_cast<const char *>(grad);
  const long long span = (p.B - 1) * p.s0 + (p.T - 1) * p.s1 + (p.U1 - 1) * p.s2 + p.VD;
  const bool overlap = p.B > 0 && go < lo + span * (long long)sizeof(*grad) &&
                       lo < go + p.B * p.T * p.U1 * p.VD * (long long)sizeof(*grad);
  // one layout for logits and gradient, at the same offset from a 16-byte
  // boundary: every row takes the aligned vector path
  const bool same_layout = p.s2 == p.VD && p.s1 == p.U1 * p.VD && p.s0 == p.T * p.s1 &&
                           ((reinterpret_cast<uintptr_t>(lo) - reinterpret_cast<uintptr_t>(go)) &
                            15) == 0;
  // (an output that overlaps the logits is the contiguous logits themselves:
  // the argument checks reject any other overlap)
  // staged rows (chunks to shared memory by cp.async): realigned long rows
  // of a strided view, and fp32 rows of one contiguous layout; never when
  // writing in place.  Measured per step: parakeet 0.4995 vs 0.5096 ms,
  // long_labels 3.485 vs 3.519 ms; contiguous bf16 rows were slower staged
  // (large_batch 1.576 vs 1.519 ms) and keep the register batches.
  const bool stage = !overlap && (same_layout ? DT == kF32 : TPR == kStagedViewTPR);
  auto kern = overlap       ? grad_kernel<DT, TPR, true, false, false>
              : same_layout ? (stage ? grad_kernel<DT, TPR, false, false, true>
                                     : grad_kernel<DT, TPR, false, false, false>)
                            : (stage ? grad_kernel<DT, TPR, false, true, true>
                                     : grad_kernel<DT, TPR, false, true, false>);
  // staged rows keep their chunks in the dynamic shared memory (the
  // streaming passes request at least kStreamSmemReserve anyway)
  size_t smem = kStreamSmemReserve;
  if (stage) {
    const size_t st = (size_t)RPB * 16 * stage_chunks(p.V * (long long)sizeof(*grad));
    if (st > smem) smem = st;
    if (smem > 48 * 1024) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
  }
  kern<<<(unsigned)blocks, kGradThreads, smem, stream>>>(p, ws, grad, gscale, n_begin, n_end);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const Problem &p, const Workspace &ws, void *grad_out, const float *gscale,
                      long long n_begin, long long n_end, cudaStream_t stream) {
  typedef typename Elem<DT>::T E;
  E *g = static_cast<E *>(grad_out);
  const long long row_bytes = p.V * (long long)sizeof(E);
  int tpr =
      row_bytes >= kLongRowBytes ? 256 : row_group_threads(row_bytes, kVecPerThread);
  // Long rows of a strided view whose rows sit at other 16-byte offsets than
  // the gradient rows (the staged realigned path): 64 lanes per row, four
  // rows per block (measured on the bf16 [..., :8198] view of [..., 8205],
  // ragged: 0.2585-0.2592 ms per step, against 0.263 with 128 lanes and
  // 0.291 with 256)
  if (tpr == 256) {
    const char *lo = static_cast<const char *>(p.logits);
    const bool same_layout =
        p.s2 == p.VD && p.s1 == p.U1 * p.VD && p.s0 == p.T * p.s1 &&
        ((reinterpret_cast<uintptr_t>(lo) - reinterpret_cast<uintptr_t>(g)) & 15) == 0;
    if (!same_layout) tpr = kStagedViewTPR;
  }
  switch (tpr) {
    case 8: return launch_tpr<DT, 8>(p, ws, g, gscale, n_begin, n_end, stream);
    case 16: return launch_tpr<DT, 16>(p, ws, g, gscale, n_begin, n_end, stream);
    case 32: return launch_tpr<DT, 32>(p, ws, g, gscale, n_begin, n_end, stream);
    case 64: return launch_tpr<DT, 64>(p, ws, g, gscale, n_begin, n_end, stream);
    case 128: return launch_tpr<DT, 128>(p, ws, g, gscale, n_begin, n_end, stream);
    default: return launch_tpr<DT, 256>(p, ws, g, gscale, n_begin, n_end, stream);
  }
}

}  // namespace

cudaError_t launch_grad(const Problem &p, int dtype, const Workspace &ws, void *grad_out,
                        const float *gscale, long long n_begin, long long n_end,
                        cudaStream_t stream) {
  if (n_end - n_begin <= 0) return cudaSuccess;
  switch (dtype) {
    case kF32: return launch_dt<kF32>(p, ws, grad_out, gscale, n_begin, n_end, stream);
    case kF16: return launch_dt<kF16>(p, ws, grad_out, gscale, n_begin, n_end, stream);
    default: return launch_dt<kBF16>(p, ws, grad_out, gscale, n_begin, n_end, stream);
  }
}

}  // namespace tdt
