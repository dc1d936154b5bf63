// tdt_common.cuh -- definitions shared by the TDT loss kernels (sm_103a).
//
// Numeric representation of the lattice.  The node tables first form each
// arc's log-weight in 64-bit fixed point with 32 fraction bits ("fx": value
// * 2^32, rounded) from the fp32 logits and log-sum-exps, then store the arc
// probability as an extended-range float ("xf", struct LV): s * 2^e with an
// int32 exponent e and an fp32 mantissa s in [1, 2) (s = 0: probability 0).
// alpha, beta and the likelihood are xf values too, so the recursions run in
// the probability domain, as sums of products of positive numbers:
//   e_j = e_src + e_w                       exact integer add
//   E   = max_j e_j                         exact integer max
//   S   = sum_j (s_src s_w) 2^(e_j - E)     fp32; the scale is an exact power
//                                           of two (0 below 2^-126 of the max)
//   (e, s) = (E + x, S / 2^x)               x = exponent bits of S (exact)
// The integer exponent carries the range, so nothing underflows however long
// the chain ("float64 accumulation for precision on long label sequences",
// "tdt-loss: add TDT loss kernel", kernels-community PR #882, "What's in
// it"), and the only roundings per node are one fp32 multiply and one add
// per arc: no exponential, logarithm, conversion or division.  GB300 runs
// float64 at a small fraction of its fp32 rate, which is why the arithmetic
// is integer + fp32 rather than float64.  |e| < 2^27 for every non-zero
// value because log-probs are clamped at -4096, |sigma| <= 1024 and
// T + U + 1 <= 65536.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tdt {

typedef long long fx_t;

constexpr double kFxOne = 4294967296.0;                     // 2^32
constexpr float kLogProbFloor = -4096.0f;
// ln 2 in fx, rounded from the mathematical constant 0.693147180559945309...
constexpr fx_t kFxLn2 = (fx_t)(0.69314718055994530942 * 4294967296.0 + 0.5);
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxDurations = 32;
constexpr int kMaxDurationValue = 255;

enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum Reduction { kNone = 0, kSum = 1, kMean = 2, kMeanBatch = 3, kMeanVolume = 4 };

// Everything a kernel needs to know about one call.  Passed by value.
struct Problem {
  const void *logits;
  long long B, T, U1, VD, V, D;   // U1 = U + 1; D: duration logits per row
  long long s0, s1, s2;           // element strides of logits (s3 == 1)
  const long long *labels;        // [B, U1-1]
  const long long *logit_lens;    // [B]
  const long long *label_lens;    // [B]
  int dur[kMaxDurations];         // lattice durations
  int n_dur;
  int max_dur;
  int blank;
  int reduction;
  fx_t sigma_fx;
  long long n_diag;               // T + U1 - 1 anti-diagonals per utterance
  int rec_len;                    // fx values per node arc record (arc_record_len)
  int rnnt;                       // 1: plain RNN-T: no duration logits (D = 0); the
                                  //    lattice durations are {0, 1} with blank arcs
                                  //    of duration 1 and label arcs of duration 0 only
  long long wait_limit;           // clock cycles a lattice band waits for a neighbour
                                  //    before it gives up (set by launch_lattice)
  long long fault_utt;            // testing: the utterance whose band 1 never publishes
                                  //    its boundary row (-1: none; set by launch_lattice)
  unsigned divT_m, divU1_m;       // n / T and n / U1 for n < 2^31 as (n m) >> s
  int divT_s, divU1_s;            //    (set by the host, fast_div_setup)
  int gx_rows;                    // > 0: the lattice bands of this launch hold gx_rows
                                  //    rows each and exchange their boundary rows
                                  //    through global memory (set by the host with
                                  //    lattice_global_rows before the node tables)
};

// Division of n < 2^31 by an invariant d >= 1 with one 32 x 32 -> 64-bit
// multiply and a shift: with l = ceil(log2 d), m = floor(2^(31+l) / d) + 1
// (< 2^32) and s = 31 + l, floor(n / d) = (n m) >> s for every n < 2^31
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994).
inline void fast_div_setup(long long d, unsigned *m, int *s) {
  int l = 0;
  while ((1LL << l) < d) ++l;
  *s = 31 + l;
  *m = (unsigned)(((unsigned long long)1 << *s) / (unsigned long long)d + 1ull);
}
__device__ __forceinline__ unsigned fast_div(unsigned n, unsigned m, int s) {
  return (unsigned)(((unsigned long long)n * m) >> s);
}

// Node arc record (fx values), one per lattice node in anti-diagonal order:
//   [i] = lpB - sigma + lpD_i      blank arc with duration i
//   [D + i] = lpL - sigma + lpD_i  label arc with duration i (lpL taken as 0
//                                  where no label arc leaves the node)
// so a lattice pass adds one value per arc; 2D values = a 16-byte multiple.
__host__ __device__ inline int arc_record_len(int n_dur) { return 2 * n_dur; }

// Shared memory a K1/K4 block reserves without using it: with it, no K1/K4
// block fits beside a lattice block (which requests at least
// kLatticeSmemFloor), so the latency-bound lattice passes get SMs of their own.
constexpr int kStreamSmemReserve = 32 * 1024;
constexpr int kLatticeSmemFloor = 200 * 1024;

// A lattice value or arc probability s * 2^e (xf), 8 bytes so that one
// aligned load moves both parts; zero is s = 0, e = kXeZero.
struct __align__(8) LV {
  int e;
  float s;
};
// Exponent of a zero value: far below every non-zero value (|e| < 2^27), and
// two of them added to a third stay in int32.
constexpr int kXeZero = -(1 << 28);
// A boundary-row entry that its band has not written yet (the node-table
// pass sets the entries that lattice bands exchange to it).  Its exponent
// is one no value has (|e| < 2^27, zero is e = kXeZero), and its mantissa
// is 0, which a stored value has only together with e = kXeZero.  So a
// reader that sees either half of the marker -- even next to the other half
// of a new value -- knows the entry is not complete (lv_written).
constexpr int kXeUnwritten = (int)0x80000000;
__host__ __device__ inline LV lv_unwritten() {
  LV v;
  v.e = kXeUnwritten;
  v.s = 0.0f;
  return v;
}
__host__ __device__ inline bool lv_written(const LV &v) {
  return v.e != kXeUnwritten && (v.s != 0.0f || v.e == kXeZero);
}

// Scratch layout (device pointers carved from one workspace block).
struct Workspace {
  // anti-diagonal-major, node index g = (b * n_diag + t + u) * U1 + u
  LV *arcw;      // [g][rec_len] node arc records (arc_record_len): probabilities
  LV *alpha;     // [g]
  LV *beta;      // [g]
  float *frac;   // [g][2 + n_dur]: share of beta(t,u) through its blank arcs,
                 //   its label arcs, and through each duration (a record per
                 //   node, so the nodes of a diagonal write adjacent records)
  // node-major per-row data, index n = (b * T + t) * U1 + u
  float *lse_tok;  // log-sum-exp of the token logits
  float *lse_dur;  // log-sum-exp of the duration logits
  // per utterance
  LV *loglik;      // [B] log-likelihood from alpha (s = 0: no path)
  float *scale;    // [B] c_b, factor of dL_b/dz in the reduced loss
  int *usable;     // [B] 1 = usable: set to 1 by the node-table pass of the
                   //   utterance's chunk, cleared by the lattice passes when the
                   //   lengths or labels are unusable or a bounded wait gave up
  int *ticket;     // [B] start-order counter of the lattice launch whose first
                   //   utterance is b (global-exchange bands), zeroed by the
                   //   node-table pass
};

__host__ __device__ inline long long diag_index(const Problem &p, long long b, long long t,
                                                long long u) {
  return (b * p.n_diag + t + u) * p.U1 + u;
}

// (b, t, u) of node n = (b * T + t) * U1 + u with 32-bit divisions (64-bit
// ones are long software sequences); B * T * U1 < 2^31 is checked on the host.
__device__ __forceinline__ void decode_node(const Problem &p, long long n, long long *b,
                                            long long *t, long long *u) {
  const unsigned nn = (unsigned)n, U1 = (unsigned)p.U1, T = (unsigned)p.T;
  const unsigned bt = fast_div(nn, p.divU1_m, p.divU1_s);
  *u = nn - bt * U1;
  const unsigned bb = fast_div(bt, p.divT_m, p.divT_s);
  *t = bt - bb * T;
  *b = bb;
}

// ---- element access -------------------------------------------------------
template <int DT> struct Elem;
template <> struct Elem<kF32> {
  typedef float T;
  static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
  static __device__ __forceinline__ float to_float(float v) { return v; }
  static __device__ __forceinline__ float from_float(float v) { return v; }
};
template <> struct Elem<kF16> {
  typedef __half T;
  static __device__ __forceinline__ float load(const __half *p) { return __half2float(__ldg(p)); }
  static __device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_float(float v) { return __float2half_rn(v); }
};
template <> struct Elem<kBF16> {
  typedef __nv_bfloat16 T;
  static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
    return __bfloat162float(__ldg(p));
  }
  static __device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_float(float v) {
    return __float2bfloat16_rn(v);
  }
};

// ---- arithmetic helpers -----------------------------------------------------
// 2^x for x <= 0 (and moderate positive x) with the hardware approximation
// (ex2.approx, ~2 ulp); large negative x flush to 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fx value of a float (exact for |x| >= 2^-8 up to 2^30).
__device__ __forceinline__ fx_t fx_from_float(float x) {
  return __float2ll_rn(x * 4294967296.0f);
}

// ---- extended-range floats (xf) -------------------------------------------
__device__ __forceinline__ LV xf_zero() {
  LV v;
  v.e = kXeZero;
  v.s = 0.0f;
  return v;
}

// 2^k for k <= 0 as an exact fp32 power of two; 0 below 2^-126.
__device__ __forceinline__ float pow2_nonpos(int k) {
  return __int_as_float(max(k + 127, 0) << 23);
}

// The xf value of an unnormalised sum S around the exponent E (S * 2^E):
// the exponent bits of S move into e, the mantissa stays.  S = 0: zero.
// Every sum of arc terms taken relative to its largest exponent is >= 1.
__device__ __forceinline__ LV xf_from_sum(float S, int E) {
  if (!(S > 0.0f)) return xf_zero();
  const int bits = __float_as_int(S);
  LV v;
  v.e = E + ((bits >> 23) - 127);
  v.s = __int_as_float((bits & 0x007fffff) | 0x3f800000);
  return v;
}

// log2(e) * 2^62 rounded to an integer (6653256548922161245.87...).
constexpr long long kLog2eQ62 = 6653256548922161246LL;

// xf value of exp(w / 2^32) for an fx log-weight w (|w| < 2^62).  The base-2
// logarithm w log2(e) / 2^32 comes out of one signed 64 x 64-bit high
// product as fixed point with 30 fraction bits (error < 2^-30): its integer
// part is the exponent, its fraction goes through exp2f.
__device__ __forceinline__ LV xf_from_fx(fx_t w) {
  const long long h = __mul64hi(w, kLog2eQ62);  // floor(log2(p) * 2^30)
  LV v;
  v.e = (int)(h >> 30);
  v.s = exp2f((float)(int)(h & 0x3fffffffLL) * (1.0f / 1073741824.0f));
  if (v.s >= 2.0f) {  // a fraction within 2^-25 of 1 rounded up
    v.s *= 0.5f;
    v.e += 1;
  }
  return v;
}

__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- host side shared by the entry points (tdt_api.cu) ----------------------
struct Layout {  // byte offsets of the scratch regions inside one block
  size_t arcw, alpha, beta, lse_tok, lse_dur, frac, loglik, scale, usable, ticket, total;
};
bool make_layout(const int64_t sizes[4], int n_dur, Layout *L);
Workspace carve(const Layout &L, void *base);
int validate(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
             const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
             const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
             const float *loss_out, const void *grad_out, Problem *p, bool need_loss,
             bool rnnt = false);

// ---- launchers (one per translation unit) ----------------------------------
// Rows are flat node ids n in [n_begin, n_end); utterances b in [b_begin, b_end).
cudaError_t launch_node_tables(const Problem &p, int dtype, const Workspace &ws,
                               long long n_begin, long long n_end, cudaStream_t stream);
// started (optional): an event recorded once every block of the lattice
// launch has begun (a launch-completion event); *started_used tells whether
// it was attached (the plain fallback kernels and launches of more than
// 65535 utterances do not record it).
// Rows per band when the lattice of a launch of nb utterances splits into
// bands exchanging through global memory, else 0.  The caller stores it in
// Problem::gx_rows before the node-table pass of those utterances (which
// clears the boundary rows and the start counter) and passes the same
// Problem to launch_lattice.
int lattice_global_rows(const Problem &p, long long nb);
cudaError_t launch_lattice(const Problem &p, const Workspace &ws, long long b_begin,
                           long long b_end, bool with_beta, cudaStream_t stream,
                           cudaEvent_t started = nullptr, bool *started_used = nullptr);
cudaError_t launch_reduce(const Problem &p, const Workspace &ws, float *loss_out,
                          cudaStream_t stream);
// gscale: device upstream gradient of the loss ([B] for kNone, else [1]) or NULL (= 1)
cudaError_t launch_grad(const Problem &p, int dtype, const Workspace &ws, void *grad_out,
                        const float *gscale, long long n_begin, long long n_end,
                        cudaStream_t stream);
}  // namespace tdt
