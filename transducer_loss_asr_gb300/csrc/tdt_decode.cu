// tdt_decode.cu -- greedy TDT decoding over precomputed joint outputs.
//
// "Add TDT loss kernel" (transformers PR #46048), commit list: greedy TDT
// decoding with per-token timestamps and token durations, and a guard on
// the symbols emitted per frame (max_symbols_per_step).  Given the joint
// output z[b, t, u, :] for every frame t and decoder state u, utterance b
// is decoded by the walk
//   t = u = 0; at (t, u): k = first argmax of z[0:V), d = durations[first
//   argmax of z[V:V+D)]; a token k != blank is emitted with frame t and
//   duration d and u advances (decoding stops when no row u is left); a
//   blank, or a token once max_symbols tokens were emitted at this frame,
//   moves at least one frame; otherwise t advances by d; stop at t >= T_b.
// One CTA per utterance: each step the CTA takes a block-wide argmax of the
// row (smallest index among equal maxima, values compared in fp32 after an
// exact conversion from the input dtype), and thread 0 takes the step.
// Every step advances t or u, so an utterance takes at most T_b + U + 1
// steps; the loop is bounded by that.
#include <climits>

#include "../../include/tdt_loss.h"
#include "tdt_rowio.cuh"

namespace tdt {

namespace {

constexpr int kDecodeThreads = 256;

struct DecodeArgs {
  const void *logits;
  long long T, U1, V, D;
  long long s0, s1, s2;
  const long long *logit_lens;
  int dur[kMaxDurations];
  int blank, max_symbols;
  int *n_out, *tokens, *frames, *durs;  // [B], [B][U1] x 3
};

__device__ __forceinline__ void keep_better(float &bv, int &bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

// Block-wide argmax; the result is valid in thread 0.  Every thread calls it.
__device__ void block_argmax(float &v, int &i, float *sv, int *si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    keep_better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = v;
    si[warp] = i;
  }
  __syncthreads();
  if (warp == 0) {
    v = lane < kDecodeThreads / 32 ? sv[lane] : -INFINITY;
    i = lane < kDecodeThreads / 32 ? si[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      keep_better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  }
  __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(kDecodeThreads) greedy_decode_kernel(DecodeArgs a) {
  typedef typename Elem<DT>::T E;
  __shared__ float sv[kDecodeThreads / 32];
  __shared__ int si[kDecodeThreads / 32];
  __shared__ int s_t, s_u, s_done;
  const long long b = blockIdx.x;
  const E *logits = static_cast<const E *>(a.logits);
  const long long Tb = a.logit_lens[b];
  int *tok = a.tokens + b * a.U1, *frm = a.frames + b * a.U1, *dus = a.durs + b * a.U1;
  int n = 0, here = 0;  // thread 0's counters
  if (threadIdx.x == 0) {
    s_t = 0;
    s_u = 0;
    s_done = (Tb < 1 || Tb > a.T) ? 1 : 0;  // unusable length: nothing decoded
  }
  __syncthreads();
  const long long max_steps = (Tb > 0 ? Tb : 0) + a.U1 + 1;
  for (long long step = 0; step < max_steps; ++step) {
    if (s_done) break;
    const int t = s_t, u = s_u;
    const E *row = logits + b * a.s0 + (long long)t * a.s1 + (long long)u * a.s2;
    float v = -INFINITY;
    int k = INT_MAX;
    for (long long j = threadIdx.x; j < a.V; j += kDecodeThreads)
      keep_better(v, k, Elem<DT>::to_float(row[j]), (int)j);
    block_argmax(v, k, sv, si);
    float vd = -INFINITY;
    int id = INT_MAX;
    if (threadIdx.x < a.D) keep_better(vd, id, Elem<DT>::to_float(row[a.V + threadIdx.x]),
                                       (int)threadIdx.x);
    block_argmax(vd, id, sv, si);
    if (threadIdx.x == 0) {
      // an all-NaN part has no maximum: take index 0 (logits are meant to be finite)
      if (k == INT_MAX) k = 0;
      if (id == INT_MAX) id = 0;
      int d = a.dur[id];
      int nt = t, nu = u, done = 0;
      if (k != a.blank) {
        tok[n] = k;
        frm[n] = t;
        dus[n] = d;
        ++n;
        ++here;
        ++nu;
        if (nu >= a.U1) done = 1;  // no joint output for row U + 1
      }
      if (d == 0 && (k == a.blank || here >= a.max_symbols)) d = 1;
      if (d > 0) {
        nt += d;
        here = 0;
      }
      if (nt >= Tb) done = 1;
      s_t = nt;
      s_u = nu;
      s_done = done;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.n_out[b] = n;
    s_u = n;
  }
  __syncthreads();
  for (long long j = s_u + threadIdx.x; j < a.U1; j += kDecodeThreads) {
    tok[j] = -1;
    frm[j] = -1;
    dus[j] = -1;
  }
}

}  // namespace
}  // namespace tdt

extern "C" int tdt_greedy_decode(const void *logits, const int64_t sizes[4],
                                 const int64_t strides[4], int dtype, const int64_t *logit_lens,
                                 const int32_t *durations, int n_dur, int blank, int max_symbols,
                                 int32_t *n_out, int32_t *tokens_out, int32_t *frames_out,
                                 int32_t *durations_out, void *stream) {
  using namespace tdt;
  if (!sizes || !strides || !durations) return TDT_ERR_NULL_POINTER;
  if (dtype != TDT_DTYPE_F32 && dtype != TDT_DTYPE_F16 && dtype != TDT_DTYPE_BF16)
    return TDT_ERR_BAD_DTYPE;
  if (n_dur < 1 || n_dur > kMaxDurations) return TDT_ERR_BAD_DURATIONS;
  const long long B = sizes[0], T = sizes[1], U1 = sizes[2], VD = sizes[3];
  if (B < 0 || T < 1 || U1 < 1 || VD <= n_dur || B > 2147483647LL) return TDT_ERR_BAD_SIZES;
  if (T >= (1LL << 30) || U1 >= (1LL << 30)) return TDT_ERR_BAD_SIZES;
  if (strides[3] != 1 || strides[0] < 0 || strides[1] < 0 || strides[2] < 0)
    return TDT_ERR_BAD_STRIDES;
  for (int i = 0; i < n_dur; ++i)
    if (durations[i] < 0 || durations[i] > kMaxDurationValue) return TDT_ERR_BAD_DURATIONS;
  const long long V = VD - n_dur;
  if (blank < 0 || blank >= V) return TDT_ERR_BAD_BLANK;
  if (max_symbols < 1) return TDT_ERR_BAD_SIZES;
  if (B == 0) return TDT_OK;
  if (!logits || !logit_lens || !n_out || !tokens_out || !frames_out || !durations_out)
    return TDT_ERR_NULL_POINTER;
  const size_t es = dtype == TDT_DTYPE_F32 ? 4 : 2;
  if (((uintptr_t)logits % es) != 0) return TDT_ERR_BAD_ALIGNMENT;
  DecodeArgs a;
  a.logits = logits;
  a.T = T;
  a.U1 = U1;
  a.V = V;
  a.D = n_dur;
  a.s0 = strides[0];
  a.s1 = strides[1];
  a.s2 = strides[2];
  a.logit_lens = reinterpret_cast<const long long *>(logit_lens);
  for (int i = 0; i < kMaxDurations; ++i) a.dur[i] = i < n_dur ? durations[i] : 0;
  a.blank = blank;
  a.max_symbols = max_symbols;
  a.n_out = n_out;
  a.tokens = tokens_out;
  a.frames = frames_out;
  a.durs = durations_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case TDT_DTYPE_F32:
      greedy_decode_kernel<kF32><<<(unsigned)B, kDecodeThreads, 0, s>>>(a);
      break;
    case TDT_DTYPE_F16:
      greedy_decode_kernel<kF16><<<(unsigned)B, kDecodeThreads, 0, s>>>(a);
      break;
    default:
      greedy_decode_kernel<kBF16><<<(unsigned)B, kDecodeThreads, 0, s>>>(a);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? TDT_OK : TDT_ERR_CUDA;
}
