// tdt_lattice.cu -- K2 alpha, K3 beta (+ arc fractions), K5 reduction.
//
// "alpha/beta passes over the lattice (float64 accumulation for precision on
// long label sequences, no 1024-label limit)" ("tdt-loss: add TDT loss
// kernel", kernels-community PR #882, "What's in it").  alpha(t,u) depends on
// (t-d,u) for d > 0 and on (t-d,u-1) for every d including 0, so all of its
// inputs lie on earlier anti-diagonals t+u: the passes walk the
// anti-diagonals (in reverse for beta), one barrier per diagonal.  Arc
// weights, alpha and beta are probabilities held as extended-range floats
// s * 2^e (int32 exponent, fp32 mantissa; tdt_common.cuh), so a node's value
// is a plain sum of products.  alpha and beta are also stored in global
// memory in the anti-diagonal layout for the gradient pass.
//
// Two variants:
//  * lattice_cluster_kernel (D <= 9): the rows u of an utterance's lattice
//    are split into K bands, one CTA each, the K CTAs of an utterance and
//    direction forming a thread-block cluster.  G lanes serve one node (one
//    up to five durations, else two; lane k takes durations k, k+G, ...).
//    A CTA keeps the values of the last RA
//    diagonals of its rows in a shared ring, and the arc records of the
//    diagonals in flight in a second ring filled with cp.async P diagonals
//    ahead (with several bands by the control warp, a diagonal's records of
//    the band's rows being one contiguous block in the anti-diagonal layout;
//    with one band by each node's lanes), so no global round trip sits on
//    the diagonal-to-diagonal path.  K: one band up to 16 compute warps,
//    else as many bands as a cluster allows (then the fewest whose rings
//    fit).  With K = 1 the kernel is compiled without any exchange.
//    With K > 1 the one row a band needs from its neighbour (u_lo - 1 for
//    alpha, u_hi + 1 for beta) is pushed into the neighbour's ring through
//    distributed shared memory after every diagonal (st.async counted on an
//    mbarrier per ring slot), and a second mbarrier per slot says "consumed",
//    so neighbouring bands run a few diagonals apart with no cluster-wide
//    barrier per diagonal.  Every wait is bounded: past the limit the
//    utterance is marked unusable (NaN loss) and the CTA stops.
//    Lattices too tall for one CTA instead split into many small bands (as
//    many as a 128-CTA launch allows: long_labels, 1,201 rows, takes 64 of
//    19 rows per direction) that are not a cluster: a band's boundary row
//    goes to its neighbour through global memory.  The node-table pass
//    clears those boundary entries to a marker no lattice value has
//    (lv_unwritten); node values are stored with gpu-scope relaxed 64-bit
//    stores, and one thread of the consuming band copies each boundary
//    value into its ring with the arc records, checks it a step before it
//    is needed and polls (bounded) only if it was not written yet.  CTAs
//    take their band from a start-order ticket, so a band only waits on
//    bands that started before it.
//  * alpha_kernel / beta_kernel: the same wavefront reading and writing
//    global memory, any U and D (no limit on label length).
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "tdt_async.cuh"
#include "tdt_common.cuh"

namespace tdt {

extern __shared__ __align__(16) unsigned char tdt_dyn_smem[];

// Band count forced by tdt_loss_set_lattice_bands (0: chosen per problem).
std::atomic<int> g_forced_bands{0};
// How bands exchange boundary rows, forced by tdt_loss_set_lattice_exchange
// (0: chosen per problem, 1: thread-block cluster, 2: global memory).
std::atomic<int> g_forced_exchange{0};
// Testing support (tdt_loss_test_set_halo_fault): the utterance whose band 1
// withholds its boundary row (-1: none) and the wait limit in clock cycles
// (0: kWaitLimitCycles).
std::atomic<long long> g_fault_utt{-1};
std::atomic<long long> g_wait_limit{0};

namespace {

constexpr int kLatticeMaxThreads = 1024;
// A single band holds at most 16 warps (more are split into bands), so its
// kernel may use up to 128 registers per thread.
constexpr int kLatticeOneBandThreads = 512;

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

// Per-utterance outputs of the alpha side: c_b, and the usable flag cleared
// for unusable lengths or labels (the node-table pass set it to 1 before this
// launch; a pass whose bounded wait gives up also clears it, so the flag is
// only ever cleared here, whatever order the clusters run in).
__device__ void write_utterance_info(const Problem &p, const Workspace &ws, long long b, bool ok,
                                     double sum_u) {
  if (!ok) ws.usable[b] = 0;
  double c = 1.0;
  if (p.reduction == kMean) c = 1.0 / ((double)p.B * (double)p.label_lens[b]);
  else if (p.reduction == kMeanBatch) c = 1.0 / (double)p.B;
  else if (p.reduction == kMeanVolume) c = 1.0 / sum_u;
  ws.scale[b] = (float)c;
  if (!ok) ws.loglik[b] = xf_zero();
}

// Sum of n candidate arc terms S_j 2^E_j (S_j = 0, E_j = kXeZero: no arc)
// as an xf value; with term non-null also each term scaled to the largest
// exponent and 1 / their sum (n <= 2 * kMaxDurations).
__device__ LV sum_terms_n(const int *E, const float *S, int n, float *term, float *inv_total) {
  int emax = E[0];
  for (int j = 1; j < n; ++j) emax = max(emax, E[j]);
  float tot = 0.0f;
  for (int j = 0; j < n; ++j) {
    const float x = S[j] * pow2_nonpos(E[j] - emax);
    if (term) term[j] = x;
    tot += x;
  }
  if (inv_total) *inv_total = tot > 0.0f ? fast_rcp(tot) : 0.0f;
  return xf_from_sum(tot, emax);
}

__device__ __forceinline__ LV xf_one() {
  LV v;
  v.e = 0;
  v.s = 1.0f;
  return v;
}

// log-likelihood: a blank arc from (T_b - d, U_b) lands exactly on T_b.
// Reads alpha and the arc weights from global memory (one thread).
__device__ void termination(const Problem &p, const Workspace &ws, long long b, long long Tb,
                            long long Ub) {
  int E[kMaxDurations];
  float S[kMaxDurations];
  for (int i = 0; i < p.n_dur; ++i) {
    const int d = p.dur[i];
    E[i] = kXeZero;
    S[i] = 0.0f;
    if (d <= 0 || Tb - d < 0) continue;
    const long long g = diag_index(p, b, Tb - d, Ub);
    const LV a = ws.alpha[g], w = ws.arcw[g * p.rec_len + i];
    E[i] = a.e + w.e;
    S[i] = a.s * w.s;
  }
  ws.loglik[b] = sum_terms_n(E, S, p.n_dur, nullptr, nullptr);
}

// Shares of beta(t,u) through blank arcs, label arcs and each duration (arc
// posteriors divided by the node occupancy), from the per-arc terms, into
// the fraction record of anti-diagonal slot g.
__device__ __forceinline__ void write_fractions(const Workspace &ws, long long g,
                                                const float *term, float inv, int nd) {
  float *fr = ws.frac + g * (2 + nd);
  float fb = 0.0f, fl = 0.0f;
  for (int i = 0; i < nd; ++i) {
    fb += term[i];
    fl += term[nd + i];
    fr[2 + i] = (term[i] + term[nd + i]) * inv;
  }
  fr[0] = fb * inv;
  fr[1] = fl * inv;
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
      LV v = xf_one();
      if (s > 0) {
        int E[2 * kMaxDurations];
        float S[2 * kMaxDurations];
        for (int i = 0; i < nd; ++i) {
          const int d = p.dur[i];
          E[i] = E[nd + i] = kXeZero;
          S[i] = S[nd + i] = 0.0f;
          if (t - d < 0) continue;
          if (d > 0) {
            const long long g = diag_index(p, b, t - d, u);
            const LV a = ws.alpha[g], w = ws.arcw[g * p.rec_len + i];
            E[i] = a.e + w.e;
            S[i] = a.s * w.s;
          }
          if (u >= 1) {
            const long long g = diag_index(p, b, t - d, u - 1);
            const LV a = ws.alpha[g], w = ws.arcw[g * p.rec_len + nd + i];
            E[nd + i] = a.e + w.e;
            S[nd + i] = a.s * w.s;
          }
        }
        v = sum_terms_n(E, S, 2 * nd, nullptr, nullptr);
      }
      ws.alpha[diag_index(p, b, t, u)] = v;
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
      const LV *rec = ws.arcw + q * p.rec_len;
      int E[2 * kMaxDurations];
      float S[2 * kMaxDurations], term[2 * kMaxDurations];
      for (int i = 0; i < nd; ++i) {
        const int d = p.dur[i];
        E[i] = E[nd + i] = kXeZero;
        S[i] = S[nd + i] = 0.0f;
        if (d > 0) {
          if (t + d < Tb) {
            const LV bb = ws.beta[diag_index(p, b, t + d, u)];
            E[i] = bb.e + rec[i].e;
            S[i] = bb.s * rec[i].s;
          } else if (t + d == Tb && u == Ub) {
            E[i] = rec[i].e;
            S[i] = rec[i].s;
          }
        }
        if (u < Ub && t + d < Tb) {
          const LV bb = ws.beta[diag_index(p, b, t + d, u + 1)];
          E[nd + i] = bb.e + rec[nd + i].e;
          S[nd + i] = bb.s * rec[nd + i].s;
        }
      }
      float inv;
      const LV v = sum_terms_n(E, S, 2 * nd, term, &inv);
      write_fractions(ws, q, term, inv, nd);
      ws.beta[q] = v;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- cluster variant

// Diagonals of arc records copied ahead of use: kPrefetchDeep when the
// record ring fits (single band), else kPrefetch.  At ~0.5-1 us per
// diagonal either covers the L2/HBM latency; the deeper one also covers it
// while the streaming passes load HBM.  Global-exchange bands whose launch
// covers the whole batch take kPrefetchShort: nothing else runs beside
// such a launch (the node tables are done, the gradient waits for it), and
// a shorter lead shortens the chain's start-up lag (long_labels lattice
// 1.614 vs 1.665 ms).
constexpr int kPrefetch = 4;
constexpr int kPrefetchDeep = 8;
constexpr int kPrefetchShort = 2;

// ---- cluster primitives (PTX ISA: mapa, barrier.cluster, st.async); the
// copy and mbarrier helpers are in tdt_async.cuh
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Shared-memory address, in CTA `cta` of the cluster, of the local object at p.
__device__ __forceinline__ unsigned map_cta(const void *p, unsigned cta) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(cta));
  return r;
}
// Asynchronous 8-byte store of a value into another CTA's shared memory
// that, when the bytes land, counts them on that CTA's mbarrier
// (complete_tx): no release fence, so the storing thread never waits for its
// own earlier memory traffic.
__device__ __forceinline__ void st_async_lv(unsigned addr, const LV &v, unsigned bar_addr) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
      ::"r"(addr), "r"((unsigned)v.e), "r"(__float_as_uint(v.s)), "r"(bar_addr)
      : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, relaxed: used only
// to say "slot consumed", after a CTA barrier that every reader of the slot
// reached with its loads of the slot already returned (their values feed
// the selects before the group shuffles), so no later store into the slot can
// affect them; a release here would be a cluster-scope fence per step.
__device__ __forceinline__ void arrive_cluster_relaxed(unsigned bar_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr)
               : "memory");
}
// Lanes per node: one for up to five durations (a lane takes all 2D arcs of
// its node), two above (lane k takes durations k, k + 2, ...).  With a term
// costing an integer add, a multiply and an exact scale, fewer warps per
// band beat a shorter per-lane chain until a lane holds ~10 terms.  Measured
// per diagonal, 1 / 2 / 4 / 8 lanes: parakeet (D = 5) 0.475 / 0.531 / 0.577
// / 0.524 us, large_batch (D = 5) 0.529 / 0.585 / 0.710 / 0.634 us,
// long_labels (D = 9) 0.915 / 0.853 / 0.893 / 1.058 us.
constexpr int group_lanes(int nd) { return nd <= 5 ? 1 : 2; }

// How the bands of an utterance exchange boundary rows.
enum Exchange {
  kXNone = 0,     // one band: no exchange
  kXCluster = 1,  // a thread-block cluster: distributed shared memory + mbarriers
  kXGlobal = 2,   // any number of bands: global memory, polled
};

// ---- global-memory exchange (PTX ISA memory consistency model: relaxed
// strong operations at gpu scope; an aligned 64-bit access is single-copy
// atomic, so a reader sees either the cleared word or the whole value)
// 64-bit gpu-scope relaxed store of a value if `pred` (predicated, no branch).
__device__ __forceinline__ void st_relaxed_gpu_lv_if(bool pred, LV *p, const LV &v) {
  const unsigned long long w =
      (unsigned long long)(unsigned)v.e | ((unsigned long long)__float_as_uint(v.s) << 32);
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p st.relaxed.gpu.global.b64 [%0], %1;\n\t}" ::"l"(p),
      "l"(w), "r"((int)pred)
      : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_bits(const LV *p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ LV lv_from_bits(unsigned long long w) {
  LV v;
  v.e = (int)(unsigned)w;
  v.s = __uint_as_float((unsigned)(w >> 32));
  return v;
}
// Poll the boundary-row entry at p until it is written (lv_written), for at
// most `limit` clock cycles; false on timeout.
__device__ __forceinline__ bool poll_written_bounded(const LV *p, long long limit, LV *out) {
  LV x = lv_from_bits(ld_relaxed_gpu_bits(p));
  if (lv_written(x)) {
    *out = x;
    return true;
  }
  const long long t0 = clock64();
  do {
    x = lv_from_bits(ld_relaxed_gpu_bits(p));
    if (lv_written(x)) {
      *out = x;
      return true;
    }
  } while (clock64() - t0 <= limit);
  return false;
}

// Launch-time shape of the cluster variant.
struct ClusterPlan {
  int X;        // Exchange: kXNone (K = 1), kXCluster or kXGlobal
  int dirs;     // directions per utterance in the launch (2: alpha and beta)
  int K;        // CTAs per (utterance, direction): the bands (cluster size for kXCluster)
  int Rc;       // lattice rows per CTA
  int G;        // lanes per node
  int RA, RW;   // slots of the value ring and of the record ring (powers of two)
  int P;        // prefetch distance in diagonals (kPrefetchDeep, kPrefetch or kPrefetchShort)
  int threads;  // (Rc + 1) * G rounded up to whole warps, plus a control warp for kXCluster
  size_t smem;  // shared bytes used
};

// Shared memory of one CTA (dynamic shared memory, addressed by byte offset
// from tdt_dyn_smem so every ring access is a 32-bit shared-space access):
//   A[RA][Rc + 2]  LV   ring row r holds lattice row u_lo + r - 1: r = 0 is
//                       the row below the band (alpha's halo), r = Rc + 1 the
//                       row above it (beta's halo)
//   W[RW][Rc + 1][REC]  node arc records of rows u_lo - 1 .. u_lo + Rc - 1
//   full[RA], empty[RA] mbarriers of the halo slots
template <int REC> struct ClusterRings {
  unsigned offW, offBar;  // byte offsets of W and of full[] (empty[] follows)
  int mA, mW, RA, slotA, slotW;  // masks, slot count, bytes per slot
  __device__ __forceinline__ LV &a(int q, int r) const {
    return *reinterpret_cast<LV *>(tdt_dyn_smem + (q & mA) * slotA + r * (int)sizeof(LV));
  }
  __device__ __forceinline__ const LV *w(int q, int r) const {
    return reinterpret_cast<const LV *>(tdt_dyn_smem + offW + (q & mW) * slotW +
                                        r * (REC * (int)sizeof(LV)));
  }
  __device__ __forceinline__ LV *w_mut(int q, int r) const {
    return reinterpret_cast<LV *>(tdt_dyn_smem + offW + (q & mW) * slotW +
                                  r * (REC * (int)sizeof(LV)));
  }
  __device__ __forceinline__ unsigned long long *full(int i) const {
    return reinterpret_cast<unsigned long long *>(tdt_dyn_smem + offBar) + i;
  }
  __device__ __forceinline__ unsigned long long *empty(int i) const {
    return reinterpret_cast<unsigned long long *>(tdt_dyn_smem + offBar) + RA + i;
  }
};

size_t cluster_smem_bytes(int RA, int RW, int Rc, int rec) {
  return (size_t)RA * (Rc + 2) * sizeof(LV) + (size_t)RW * (Rc + 1) * rec * sizeof(LV) +
         2 * (size_t)RA * 8;
}

// Copy the arc records of diagonal q for ring rows 0 .. Rc (lattice rows
// u_lo - 1 .. u_lo + Rc - 1) into the record ring, for the rows that are
// lattice nodes on that diagonal (0 <= q - u < T_b, u <= U_b).  In the
// anti-diagonal layout those records are one contiguous block in global
// memory, copied by the 32 lanes of one warp in 16-byte chunks.  Every lane
// of that warp commits one group per call, so its group count per step is
// uniform; the other warps issue no copies.
template <int REC>
__device__ __forceinline__ void prefetch_diag(const LV *gdiag0, const ClusterRings<REC> &r,
                                              int q, int u_lo, int Rc, int U1, int Tb, int Ub,
                                              int lane) {
  if (q >= 0 && q < Tb + Ub) {
    int u0 = u_lo - 1 > 0 ? u_lo - 1 : 0;
    int u1 = u_lo + Rc - 1 < U1 - 1 ? u_lo + Rc - 1 : U1 - 1;
    if (u0 < q - Tb + 1) u0 = q - Tb + 1;
    if (u1 > q) u1 = q;
    if (u1 > Ub) u1 = Ub;
    const int nch = u1 >= u0 ? (u1 - u0 + 1) * (REC / 2) : 0;
    const LV *src = gdiag0 + ((long long)q * U1 + u0) * REC;
    LV *dst = r.w_mut(q, u0 - (u_lo - 1));
    for (int c = lane; c < nch; c += 32) cp_async16(dst + 2 * c, src + 2 * c);
  }
  cp_async_commit();
}

// One band or global-exchange bands: each node's lanes copy the node's own
// record of diagonal q (if it is a lattice node): lane k copies the 16-byte
// chunks k, k+G, ...; every lane commits one group per call so the group
// count per step is uniform.  (Measured faster than one copying warp when
// there is no control warp.)  PRED: the copies are predicated in a fully
// unrolled loop, so lanes whose nodes are and are not lattice nodes on
// diagonal q do not diverge -- faster for global-exchange bands (long_labels
// lattice 1.61 -> 1.38 ms), slower for one band of five durations
// (parakeet 0.461 vs 0.416 us per diagonal), which keeps the branch.
template <int REC, int G, bool PRED>
__device__ __forceinline__ void prefetch_rec(const LV *gdiag0, const ClusterRings<REC> &r,
                                             int q, int u, int ring_row, int k, int Tb, int Ub,
                                             int U1, bool want) {
  const int t = q - u;
  const bool copy = want && q >= 0 && u >= 0 && u <= Ub && t >= 0 && t < Tb;
  if (PRED) {
    const LV *src = gdiag0 + ((long long)q * U1 + u) * REC;
    LV *dst = r.w_mut(q, ring_row);
    constexpr int kChunks = REC / 2;
#pragma unroll
    for (int c0 = 0; c0 < kChunks; c0 += G) {
      const int c = c0 + k;
      cp_async16_if(copy && c < kChunks, dst + 2 * c, src + 2 * c);
    }
  } else if (copy) {
    const LV *src = gdiag0 + ((long long)q * U1 + u) * REC;
    LV *dst = r.w_mut(q, ring_row);
    for (int c = k; c < REC / 2; c += G) cp_async16(dst + 2 * c, src + 2 * c);
  }
  cp_async_commit();
}

// Group-wide sum of this lane's 2J candidate terms S_j 2^E_j (masked ones:
// S_j = 0, E_j = kXeZero).  The reference is the group's largest exponent E
// (a 32-bit max, one shuffle per round), and each term is scaled by the
// exact power of two 2^(E_j - E), so the largest term keeps its mantissa
// (>= 1) and no term exceeds 4.  Returns E, the sum S (0 when every
// candidate is masked) and each candidate's scaled term.
template <int J, int G>
__device__ __forceinline__ void group_sum(const int *E, const float *S, int *ref_out,
                                          float *tot_out, float *term) {
  int emax = E[0];
#pragma unroll
  for (int j = 1; j < 2 * J; ++j) emax = max(emax, E[j]);
#pragma unroll
  for (int o = 1; o < G; o <<= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
  float tot = 0.0f;
#pragma unroll
  for (int j = 0; j < 2 * J; ++j) {
    term[j] = S[j] * pow2_nonpos(E[j] - emax);
    tot += term[j];
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  *ref_out = emax;
  *tot_out = tot;
}

// Per-CTA state shared by the two directions.
struct Band {
  int k, K;       // this CTA's band and the cluster size
  int Rc, u_lo;   // rows [u_lo, u_lo + Rc)
  int row, lane;  // this thread's ring row (0 .. Rc; larger = idle) and lane
  bool control;       // the thread of the control warp that waits and releases
  bool control_warp;  // a thread of that warp (no compute)
  bool prefetch_warp; // a thread of the warp that copies the arc records
                      // (the control warp; with one band each node's lanes
                      // copy its own record)
  int Tb, Ub, U1;
  int *abort;     // shared flag, set after the loop: a bounded wait gave up
};

// Halo protocol, per ring slot (a slot is reused every RA steps):
//   full[slot]   the neighbour's value of step j has landed: armed by this
//                CTA's control thread (arrive + expect 16 bytes), completed
//                by the neighbour's st.async (16 bytes)
//   empty[slot]  the neighbour has consumed step j: its control thread
//                arrives after the barrier that ends its last read of j
// Step j's halo value is read at steps j+1 .. j+1+max_dur, so it is released
// at step j+2+max_dur; the producer of step j waits for the release of step
// j - RA before storing.  The control warp issues no global stores and no
// compute; it copies the arc records into the record ring.

template <int ND, int G, int X, int P>
__device__ __forceinline__ void alpha_cluster(const Problem &p, const Workspace &ws,
                                              const ClusterRings<2 * ND> r, const ClusterPlan cp,
                                              const Band bd, long long b) {
  constexpr bool MULTI = X == kXCluster, GX = X == kXGlobal;
  constexpr int REC = 2 * ND;
  constexpr int J = (ND + G - 1) / G;
  const int row = bd.row, k = bd.lane;
  const int rowc = row <= cp.Rc ? row : cp.Rc;  // idle threads read in bounds
  const int rl = rowc >= 1 ? rowc - 1 : 0;
  const int u = bd.u_lo + row - 1;
  const bool own = row >= 1 && row <= cp.Rc;
  const bool lower = (MULTI || GX) && bd.k > 0, upper = (MULTI || GX) && bd.k + 1 < bd.K;
  const LV *gdiag0 = ws.arcw + b * p.n_diag * p.U1 * REC;
  LV *galpha = ws.alpha + b * p.n_diag * p.U1;
  // lane k takes durations k, k + G, ...; with G not dividing ND the last
  // slot of some lanes is idle; those and the blank arc of duration 0 are
  // masked by per-lane constants
  constexpr bool kIdle = (ND % G) != 0;
  int di[J], dd[J];
  bool live[J], liveb[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    live[j] = !kIdle || k + G * j < ND;
    di[j] = live[j] ? k + G * j : 0;
    dd[j] = live[j] ? p.dur[di[j]] : 0;
    liveb[j] = live[j] && dd[j] > 0;  // no blank arc of duration 0
  }
  const int nsteps = bd.Tb + bd.Ub;
  const bool pref = MULTI ? bd.prefetch_warp : row <= cp.Rc;
  const int plane = threadIdx.x & 31;
  // feeds the upper band (testing: band 1 of utterance fault_utt never does,
  // so the upper band's bounded wait runs out)
  const bool feeds = !(bd.k == 1 && b == p.fault_utt);
  const bool producer = MULTI && upper && row == cp.Rc && k == 0 && feeds;
  // global exchange: every node's value is stored with a gpu-scope relaxed
  // store (the upper band reads the top row's), and thread 0 (ring row 0,
  // whose lanes compute nothing they keep) copies row u_lo - 1 of the lower
  // band into ring row 0 with cp.async, P diagonals ahead in the same group
  // as the arc records.  It
  // checks diagonal s's value during step s, one step before its use,
  // reading it right after the barrier and testing it at the end of the
  // step, and polls for it only if it was not written yet when copied.
  const bool gx_top = GX && upper && row == cp.Rc && k == 0;
  const bool gx_halo = GX && lower && threadIdx.x == 0;
  const int uh = bd.u_lo - 1;  // the lower band's top row
  const LV *halo_src = galpha + uh;
  // (q, uh) is a lattice node iff its frame q - uh lies in [0, T_b)
  auto halo_node = [&](int q) { return q - uh >= 0 && q - uh < bd.Tb && uh <= bd.Ub; };
  int failed = 0;  // a bounded wait of this thread gave up
  auto prefetch = [&](int q) {
    if (MULTI) {
      if (pref) prefetch_diag<REC>(gdiag0, r, q, bd.u_lo, cp.Rc, bd.U1, bd.Tb, bd.Ub, plane);
    } else {
      // the lower band's value of diagonal q, used at step q + 1
      if (GX) cp_async8_if(gx_halo && halo_node(q), &r.a(q, 0), halo_src + (long long)q * bd.U1);
      prefetch_rec<REC, G, GX>(gdiag0, r, q, u, rowc, k, bd.Tb, bd.Ub, bd.U1, pref);
    }
  };
  for (int q = 0; q < P; ++q) prefetch(q);
  // halo slots armed ahead (arrive + expect 16 bytes): the first use of
  // every slot now, each later use right after the previous one was waited
  // for, past the barrier, so only the wait sits before it
  if (MULTI && bd.control && lower)
    for (int j = 0; j < r.RA && j <= nsteps - 2; ++j)
      arrive_expect_tx(r.full(j), (unsigned)sizeof(LV));
  for (int s = 0; s < nsteps; ++s) {
    prefetch(s + P);
    cp_async_wait<P>();
    if (MULTI && bd.control && lower && s >= 1) {
      // the lower band's value of diagonal s - 1
      if (!wait_parity_bounded(r.full((s - 1) & r.mA), ((s - 1) / r.RA) & 1, p.wait_limit))
        failed = 1;
    }
    // a thread whose wait gave up raises the CTA's abort flag before the
    // barrier (every write to it precedes one), and all leave together after
    // it; a plain barrier and a flag read cost less per diagonal than a
    // barrier with a reduction (measured: long_labels lattice 4.79 vs 4.85 ms)
    if ((MULTI || GX) && failed) *bd.abort = 1;
    __syncthreads();
    if ((MULTI || GX) && *bd.abort) break;
    // the slot of diagonal s - 1 serves diagonal s - 1 + RA next
    if (MULTI && bd.control && lower && s >= 1 && s - 1 + r.RA <= nsteps - 2)
      arrive_expect_tx(r.full((s - 1) & r.mA), (unsigned)sizeof(LV));
    // every thread is past step s - 1: release diagonal s - 2 - max_dur
    if (MULTI && bd.control && lower && s - 2 - p.max_dur >= 0)
      arrive_cluster_relaxed(map_cta(r.empty((s - 2 - p.max_dur) & r.mA), bd.k - 1));
    if (MULTI && bd.control_warp) continue;
    // the copy of the lower band's value of diagonal s is complete (every
    // thread reads it: a broadcast, and no branch)
    const LV halo_next = GX ? r.a(s, 0) : xf_zero();
    const int t = s - u;
    const bool node = own && u <= bd.Ub && t >= 0 && t < bd.Tb;
    int E[2 * J];
    float S[2 * J], term[2 * J];
    // blank arc (t-d, u) -> (t, u) and label arc (t-d, u-1) -> (t, u) of
    // every duration d, with no test per step: a missing source (before frame
    // 0, below row 0, outside the lattice) reads zero, because the rings
    // start zeroed and every slot of a non-node holds zero
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int d = dd[j], i = di[j];
      const LV ab = r.a(s - d, rowc), wb = r.w(s - d, rowc)[i];
      const LV al = r.a(s - d - 1, rl), wl = r.w(s - d - 1, rl)[ND + i];
      E[2 * j] = liveb[j] ? ab.e + wb.e : kXeZero;
      S[2 * j] = liveb[j] ? ab.s * wb.s : 0.0f;
      E[2 * j + 1] = live[j] ? al.e + wl.e : kXeZero;
      S[2 * j + 1] = live[j] ? al.s * wl.s : 0.0f;
    }
    int es;
    float tot;
    group_sum<J, G>(E, S, &es, &tot, term);
    // every lane of the group holds the node's value; lane 0 stores it
    const LV v = node ? (s == 0 ? xf_one() : xf_from_sum(tot, es)) : xf_zero();
    if (own && k == 0) r.a(s, row) = v;
    if (GX) {
      // every node's value with the same gpu-scope relaxed store (the top
      // row's are polled by the upper band), so no lane branches
      st_relaxed_gpu_lv_if(node && k == 0 && (feeds || !gx_top),
                           galpha + (long long)s * bd.U1 + u, v);
    } else if (node && k == 0) {
      galpha[(long long)s * bd.U1 + u] = v;
    }
    if (GX) {
      // ring row 0 of diagonal s, read from the next step on: the lower
      // band's value, polled for if it was not written when copied (a
      // branch of thread 0 alone, rarely taken: measured faster than a warp
      // vote around it)
      const bool hn = halo_node(s);
      if (gx_halo && !hn) r.a(s, 0) = xf_zero();
      const bool need = gx_halo && hn && !lv_written(halo_next);
      if (need) {  // thread 0 only, rarely
        LV hv;
        if (!poll_written_bounded(halo_src + (long long)s * bd.U1, p.wait_limit, &hv)) failed = 1;
        r.a(s, 0) = hv;
      }
    }
    if (producer) {
      // publish this diagonal's top row into the upper band's halo slot once
      // that band has released the slot's previous diagonal
      if (s >= r.RA &&
          !wait_parity_bounded(r.empty(s & r.mA), ((s / r.RA) - 1) & 1, p.wait_limit))
        failed = 1;
      else
        st_async_lv(map_cta(&r.a(s, 0), bd.k + 1), v, map_cta(r.full(s & r.mA), bd.k + 1));
    }
  }
  cp_async_wait<0>();
  if (MULTI || GX) {
    if (__syncthreads_or(failed) && threadIdx.x == 0) *bd.abort = 1;
  } else {
    __syncthreads();
  }
}

template <int ND, int G, int X, int P>
__device__ __forceinline__ void beta_cluster(const Problem &p, const Workspace &ws,
                                             const ClusterRings<2 * ND> r, const ClusterPlan cp,
                                             const Band bd, long long b) {
  constexpr bool MULTI = X == kXCluster, GX = X == kXGlobal;
  constexpr int REC = 2 * ND;
  constexpr int J = (ND + G - 1) / G;
  const int row = bd.row, k = bd.lane;
  const int rowc = row <= cp.Rc ? row : cp.Rc;
  const int u = bd.u_lo + row - 1;
  const bool own = row >= 1 && row <= cp.Rc;
  const bool lower = (MULTI || GX) && bd.k > 0, upper = (MULTI || GX) && bd.k + 1 < bd.K;
  const LV *gdiag0 = ws.arcw + b * p.n_diag * p.U1 * REC;
  LV *gbeta = ws.beta + b * p.n_diag * p.U1;
  float *gfrac = ws.frac + b * p.n_diag * p.U1 * (2 + ND);
  constexpr bool kIdle = (ND % G) != 0;
  int di[J], dd[J];
  bool live[J], liveb[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    live[j] = !kIdle || k + G * j < ND;
    di[j] = live[j] ? k + G * j : 0;
    dd[j] = live[j] ? p.dur[di[j]] : 0;
    liveb[j] = live[j] && dd[j] > 0;  // no blank arc of duration 0
  }
  const int nsteps = bd.Tb + bd.Ub;
  const int last = nsteps - 1;
  const bool pref = MULTI ? bd.prefetch_warp : own;
  const int plane = threadIdx.x & 31;
  // feeds the lower band (testing: band 1 of utterance fault_utt never does)
  const bool feeds = !(bd.k == 1 && b == p.fault_utt);
  const bool producer = MULTI && lower && row == 1 && k == 0 && feeds;
  // global exchange, as in the alpha pass: gpu-scope relaxed stores of
  // every node's value (the lower band reads the bottom row's), and thread 0
  // (ring row 0 is unused here) copies row u_lo + Rc of the upper band into
  // ring row Rc + 1
  const bool gx_bottom = GX && lower && row == 1 && k == 0;
  const bool gx_halo = GX && upper && threadIdx.x == 0;
  const int uh = bd.u_lo + cp.Rc;  // the upper band's bottom row
  const LV *halo_src = gbeta + uh;
  auto halo_node = [&](int q) { return q - uh >= 0 && q - uh < bd.Tb && uh <= bd.Ub; };
  int failed = 0;  // a bounded wait of this thread gave up
  auto prefetch = [&](int q) {
    if (MULTI) {
      if (pref) prefetch_diag<REC>(gdiag0, r, q, bd.u_lo, cp.Rc, bd.U1, bd.Tb, bd.Ub, plane);
    } else {
      // the upper band's value of diagonal q, used at the step of diagonal q - 1
      if (GX)
        cp_async8_if(gx_halo && halo_node(q), &r.a(q, cp.Rc + 1),
                     halo_src + (long long)q * bd.U1);
      prefetch_rec<REC, G, GX>(gdiag0, r, q, u, rowc, k, bd.Tb, bd.Ub, bd.U1, pref);
    }
  };
  // the end state (T_b, U_b), one diagonal past the last: value 1
  if (own && k == 0 && u == bd.Ub) r.a(nsteps, row) = xf_one();
  // a label arc of duration d from row u lands before T_b on diagonals q < T_b + u - d
  int lab_end[J];
#pragma unroll
  for (int j = 0; j < J; ++j) lab_end[j] = bd.Tb + u - dd[j];
  for (int i = 0; i < P; ++i) prefetch(last - i);
  // halo slots armed ahead, as in the alpha pass
  if (MULTI && bd.control && upper)
    for (int j = 0; j < r.RA && j <= nsteps - 2; ++j)
      arrive_expect_tx(r.full(j), (unsigned)sizeof(LV));
  for (int i = 0; i < nsteps; ++i) {
    const int q = last - i;
    prefetch(q - P);
    cp_async_wait<P>();
    if (MULTI && bd.control && upper && i >= 1) {
      // the upper band's value of step i - 1 (diagonal q + 1)
      if (!wait_parity_bounded(r.full((i - 1) & r.mA), ((i - 1) / r.RA) & 1, p.wait_limit))
        failed = 1;
    }
    // a thread whose wait gave up raises the CTA's abort flag before the
    // barrier (every write to it precedes one), and all leave together after
    // it; a plain barrier and a flag read cost less per diagonal than a
    // barrier with a reduction (measured: long_labels lattice 4.79 vs 4.85 ms)
    if ((MULTI || GX) && failed) *bd.abort = 1;
    __syncthreads();
    if ((MULTI || GX) && *bd.abort) break;
    // the slot of step i - 1 serves step i - 1 + RA next
    if (MULTI && bd.control && upper && i >= 1 && i - 1 + r.RA <= nsteps - 2)
      arrive_expect_tx(r.full((i - 1) & r.mA), (unsigned)sizeof(LV));
    // every thread is past step i - 1: release step i - 2 - max_dur
    if (MULTI && bd.control && upper && i - 2 - p.max_dur >= 0)
      arrive_cluster_relaxed(map_cta(r.empty((i - 2 - p.max_dur) & r.mA), bd.k + 1));
    if (MULTI && bd.control_warp) continue;
    // the copy of the upper band's value of diagonal q is complete
    const LV halo_next = GX ? r.a(q, cp.Rc + 1) : xf_zero();
    const int t = q - u;
    const bool node = own && u <= bd.Ub && t >= 0 && t < bd.Tb;
    const LV *rec = r.w(q, rowc);
    int E[2 * J];
    float S[2 * J], term[2 * J];
    // blank arc (t, u) -> (t+d, u) and label arc (t, u) -> (t+d, u+1) of
    // every duration d: a missing target (past the last frame, above row U_b,
    // outside the lattice) reads zero, and the final blank arcs land on the
    // end state (T_b, U_b), whose slot holds 1.  A label arc must land before
    // T_b (t + d < T_b, i.e. q < lab_end[j]), which also keeps it off the end
    // state.
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int d = dd[j], i = di[j];
      const LV bb = r.a(q + d, rowc), wb = rec[i];
      const LV bl = r.a(q + d + 1, rowc + 1), wl = rec[ND + i];
      const bool okl = live[j] && q < lab_end[j];
      E[2 * j] = liveb[j] ? bb.e + wb.e : kXeZero;
      S[2 * j] = liveb[j] ? bb.s * wb.s : 0.0f;
      E[2 * j + 1] = okl ? bl.e + wl.e : kXeZero;
      S[2 * j + 1] = okl ? bl.s * wl.s : 0.0f;
    }
    int es;
    float tot;
    group_sum<J, G>(E, S, &es, &tot, term);
    const float inv = tot > 0.0f ? fast_rcp(tot) : 0.0f;
    float fb = 0.0f, fl = 0.0f;
    // the node's fraction record; the nodes of a diagonal have adjacent ones
    float *fr = gfrac + ((long long)q * bd.U1 + u) * (2 + ND);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      fb += term[2 * j];
      fl += term[2 * j + 1];
      if (node && live[j]) fr[2 + di[j]] = (term[2 * j] + term[2 * j + 1]) * inv;
    }
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
      fb += __shfl_xor_sync(0xffffffffu, fb, o);
      fl += __shfl_xor_sync(0xffffffffu, fl, o);
    }
    const LV v = node ? xf_from_sum(tot, es) : xf_zero();
    if (own && k == 0) r.a(q, row) = v;
    if (node && k == 0) {
      fr[0] = fb * inv;
      fr[1] = fl * inv;
      if (!GX) gbeta[(long long)q * bd.U1 + u] = v;
    }
    // every node's value with the same gpu-scope relaxed store (the bottom
    // row's are polled by the lower band), so no lane branches
    if (GX)
      st_relaxed_gpu_lv_if(node && k == 0 && (feeds || !gx_bottom),
                           gbeta + (long long)q * bd.U1 + u, v);
    if (GX) {
      // ring row Rc + 1 of diagonal q, read from the next step on
      const bool hn = halo_node(q);
      if (gx_halo && !hn) r.a(q, cp.Rc + 1) = xf_zero();
      const bool need = gx_halo && hn && !lv_written(halo_next);
      if (need) {  // thread 0 only, rarely
        LV hv;
        if (!poll_written_bounded(halo_src + (long long)q * bd.U1, p.wait_limit, &hv)) failed = 1;
        r.a(q, cp.Rc + 1) = hv;
      }
    }
    if (producer) {
      // publish this diagonal's bottom row into the lower band's halo slot
      if (i >= r.RA &&
          !wait_parity_bounded(r.empty(i & r.mA), ((i / r.RA) - 1) & 1, p.wait_limit))
        failed = 1;
      else
        st_async_lv(map_cta(&r.a(q, cp.Rc + 1), bd.k - 1), v,
                    map_cta(r.full(i & r.mA), bd.k - 1));
    }
  }
  cp_async_wait<0>();
  if (MULTI || GX) {
    if (__syncthreads_or(failed) && threadIdx.x == 0) *bd.abort = 1;
  } else {
    __syncthreads();
  }
}

// Block: (Rc + 1) * G compute threads (rounded up to whole warps), then,
// with cluster bands, one control warp: it copies the arc records and waits
// for and releases the halo slots.
//
// Global-exchange bands (X = kXGlobal) are CTAs of a one-dimensional grid
// that take their role from a start-order ticket (an atomic counter that
// the node-table pass zeroed): ticket j of an utterance is alpha band j / 2
// or beta band K - 1 - j / 2, so a band's only producer (alpha: the band
// below, beta: the band above) has a smaller ticket, has started before it
// and is resident.  A band therefore waits only on resident CTAs that never
// wait on it: no residency assumption, whatever else runs on the GPU.
template <int ND, int G, int X, int P>
__global__ void __launch_bounds__(X == kXCluster ? kLatticeMaxThreads : kLatticeOneBandThreads, 1)
lattice_cluster_kernel(Problem p, Workspace ws, long long b0, ClusterPlan cp) {
  constexpr bool MULTI = X == kXCluster, GX = X == kXGlobal;
  constexpr int REC = 2 * ND;
  __shared__ int s_abort;
  __shared__ int s_ticket;
  long long b;
  bool is_beta;
  int kc;
  if (GX) {
    if (threadIdx.x == 0) s_ticket = atomicAdd(ws.ticket + b0, 1);
    __syncthreads();
    const int per = cp.dirs * cp.K, rem = s_ticket % per, j = cp.dirs == 2 ? rem >> 1 : rem;
    b = b0 + s_ticket / per;
    is_beta = cp.dirs == 2 && (rem & 1);
    kc = is_beta ? cp.K - 1 - j : j;
  } else {
    b = b0 + blockIdx.y;
    is_beta = blockIdx.z == 1;
    kc = MULTI ? (int)cluster_rank() : 0;
  }
  double sum_u;
  // every CTA of the cluster sees the same utterance, so all return together
  const bool ok = check_utterance(p, b, &sum_u);
  if (!is_beta && kc == 0 && threadIdx.x == 0) write_utterance_info(p, ws, b, ok, sum_u);
  if (!ok) return;
  // a global-exchange band wholly above U_b has no node and feeds no node
  if (GX && (long long)kc * cp.Rc > p.label_lens[b]) return;
  ClusterRings<REC> r;
  r.RA = cp.RA;
  r.mA = cp.RA - 1;
  r.mW = cp.RW - 1;
  r.slotA = (cp.Rc + 2) * (int)sizeof(LV);
  r.slotW = (cp.Rc + 1) * REC * 8;
  r.offW = (unsigned)(cp.RA * r.slotA);
  r.offBar = r.offW + (unsigned)(cp.RW * r.slotW);
  const int compute_threads = cp.threads - (MULTI ? 32 : 0);
  // both rings start as zeros (exponent kXeZero, mantissa 0), so arcs from
  // or to slots not yet written contribute nothing; every region is a whole
  // number of 16-byte chunks
  {
    const uint4 z = make_uint4((unsigned)kXeZero, 0u, (unsigned)kXeZero, 0u);
    uint4 *ring = reinterpret_cast<uint4 *>(tdt_dyn_smem);
    for (unsigned c = threadIdx.x; c < r.offBar / 16; c += blockDim.x) ring[c] = z;
  }
  if (threadIdx.x == 0) {
    s_abort = 0;
    if (MULTI) {
      for (int i = 0; i < cp.RA; ++i) {
        mbar_init(r.full(i), 1);
        mbar_init(r.empty(i), 1);
      }
      fence_mbar_init_cluster();
    }
  }
  // every band's barriers exist before any band signals a neighbour
  if (MULTI) cluster_sync_all();
  else __syncthreads();
  Band bd;
  bd.k = kc;
  bd.K = cp.K;
  bd.Rc = cp.Rc;
  bd.u_lo = kc * cp.Rc;
  const bool in_compute = (int)threadIdx.x < compute_threads;
  bd.row = in_compute ? (int)threadIdx.x / G : cp.Rc + 1;  // control warp: idle row
  bd.lane = in_compute ? (int)threadIdx.x % G : 0;
  bd.control = (int)threadIdx.x == compute_threads;
  bd.control_warp = !in_compute;
  bd.prefetch_warp = MULTI && !in_compute;
  bd.Tb = (int)p.logit_lens[b];
  bd.Ub = (int)p.label_lens[b];
  bd.U1 = (int)p.U1;
  bd.abort = &s_abort;
  if (!is_beta) alpha_cluster<ND, G, X, P>(p, ws, r, cp, bd, b);
  else beta_cluster<ND, G, X, P>(p, ws, r, cp, bd, b);
  __syncthreads();
  if ((MULTI || GX) && s_abort && threadIdx.x == 0) ws.usable[b] = 0;  // a wait timed out: NaN loss
  // no band leaves while a neighbour may still write into its shared memory
  if (MULTI) cluster_sync_all();
  if (!is_beta && threadIdx.x == 0 && !s_abort && bd.Ub >= bd.u_lo &&
      bd.Ub < bd.u_lo + cp.Rc)
    termination(p, ws, b, bd.Tb, bd.Ub);
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

constexpr int kMaxCluster = 16;
constexpr size_t kClusterSmemMax = 220 * 1024;

// Shape of the banded variant for this problem with K bands exchanging by
// X (K = 1: kXNone), or false.
bool cluster_plan(const Problem &p, int K, int X, ClusterPlan *cp, bool alone = false) {
  if (p.n_dur > 9) return false;
  if (K == 1) X = kXNone;
  if (K > 1 && X == kXNone) return false;
  const int G = group_lanes(p.n_dur);
  const int Rc = (int)((p.U1 + K - 1) / K);
  K = (int)((p.U1 + Rc - 1) / Rc);  // no band without rows
  const int threads = ((Rc + 1) * G + 31) / 32 * 32 + (X == kXCluster ? 32 : 0);
  if (threads > (X == kXCluster ? kLatticeMaxThreads : kLatticeOneBandThreads)) return false;
  if (X == kXCluster && K == 1) return false;
  const int rec = arc_record_len(p.n_dur);
  // value ring: max_dur + 2 diagonals in use, the rest is how far a band may
  // run ahead of the band it feeds
  const int RA = pow2_at_least(p.max_dur + 10);
  // the deeper prefetch for a single band when its record ring still fits;
  // global-exchange bands take a shorter one (kPrefetchShort when their
  // launch runs alone): a band trails the band it reads by about P
  // diagonals (its neighbour's values are copied P diagonals ahead), so the
  // last band of a chain of K starts about K P diagonal steps after the first
  const int P0 = X == kXNone ? kPrefetchDeep : (X == kXGlobal && alone ? kPrefetchShort : kPrefetch);
  for (int P : {P0, kPrefetch}) {
    const int RW = pow2_at_least(P + p.max_dur + 3);
    const size_t bytes = cluster_smem_bytes(RA, RW, Rc, rec);
    if (bytes > kClusterSmemMax) continue;
    cp->X = X;
    cp->dirs = 2;
    cp->K = K;
    cp->Rc = Rc;
    cp->G = G;
    cp->RA = RA;
    cp->RW = RW;
    cp->P = P;
    cp->threads = threads;
    cp->smem = bytes;
    return true;
  }
  return false;
}

// Bands per utterance and direction for a launch of nb utterances.  One
// band whenever it holds at most 16 warps (splitting parakeet's band in two
// made it 40% slower: the exchange costs more than the rows it saves).
// Longer utterances take as many bands as a cluster allows: the step is
// bound by issuing the work of a CTA's warps, so fewer rows per band are
// faster (long_labels, 1,201 rows: 16 bands 0.814 us per diagonal, 13 bands
// 0.853 us; fewer than 13 leave no room for the record ring).  The bands of
// a launch take an SM each, so a launch holds at most ~48 of them; the rest
// of the GPU streams K1/K4.
int preferred_bands(const Problem &p, long long nb) {
  const int forced = g_forced_bands.load();
  if (forced > 0) return forced < kMaxCluster ? forced : kMaxCluster;
  const int warps = (int)(((p.U1 + 1) * group_lanes(p.n_dur) + 31) / 32);
  if (warps <= 16) return 1;
  const long long cap = 48 / (2 * (nb > 0 ? nb : 1));
  const int K = cap > 1 ? (int)cap : 1;
  return K < kMaxCluster ? K : kMaxCluster;
}

// Lanes of a global-exchange band (before the cap below) and the CTAs of
// such a launch: as many small bands as kGlobalBandCtas SMs allow.  A
// smaller band steps a diagonal faster (long_labels, 1,201 rows, nine
// durations, per diagonal: 39 bands 0.433 us, 50 0.404, 64 0.394, 76 0.403),
// and each band takes an SM of its own, so a launch beside other passes
// keeps to fewer (large_batch's 121-row lattices stay one band: with 2-4
// global bands the lattice got faster but the step slower, 1.54-1.71 vs
// 1.44 ms).
constexpr int kGlobalBandLanes = 32;
constexpr int kGlobalBandCtas = 128;

}  // namespace

int lattice_global_rows(const Problem &p, long long nb) {
  if (p.n_dur > 9 || nb < 1) return 0;
  const int mode = g_forced_exchange.load();
  if (mode == kXCluster) return 0;
  const int G = group_lanes(p.n_dur);
  const int forced = g_forced_bands.load();
  int K;
  if (forced > 0) {
    // forced counts up to a cluster's size use a cluster unless global
    // exchange is forced too
    if (forced == 1 || (forced <= kMaxCluster && mode != kXGlobal)) return 0;
    K = forced;
  } else {
    const int warps = (int)(((p.U1 + 1) * G + 31) / 32);
    if (warps <= 16) return 0;  // one band
    const int rows = kGlobalBandLanes / G - 1;
    K = (int)((p.U1 + rows - 1) / rows);
    const long long cap = kGlobalBandCtas / (2 * nb);
    if (K > cap) K = cap > 1 ? (int)cap : 1;
    if (K < 2) return 0;
  }
  ClusterPlan cp;
  if (!cluster_plan(p, K, kXGlobal, &cp)) return 0;
  return cp.Rc;
}

namespace {

template <int ND, int G>
cudaError_t launch_cluster_g(const Problem &p, const Workspace &ws, long long b0, long long nb,
                             bool with_beta, const ClusterPlan &cp_in, cudaStream_t stream,
                             bool *placed, cudaEvent_t started, bool *started_used) {
  *placed = false;
  ClusterPlan cp = cp_in;
  cp.dirs = with_beta ? 2 : 1;
  auto kern =
      cp.X == kXCluster
          ? lattice_cluster_kernel<ND, G, kXCluster, kPrefetch>
          : cp.X == kXGlobal
                ? (cp.P == kPrefetchShort ? lattice_cluster_kernel<ND, G, kXGlobal, kPrefetchShort>
                                          : lattice_cluster_kernel<ND, G, kXGlobal, kPrefetch>)
                : (cp.P == kPrefetchDeep ? lattice_cluster_kernel<ND, G, kXNone, kPrefetchDeep>
                                         : lattice_cluster_kernel<ND, G, kXNone, kPrefetch>);
  // at least kLatticeSmemFloor, so no node-table or gradient block shares the SM
  const size_t bytes = cp.smem < (size_t)kLatticeSmemFloor ? (size_t)kLatticeSmemFloor : cp.smem;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && cp.X == kXCluster && cp.K > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  // global-exchange bands: one-dimensional, roles by start-order ticket
  const dim3 grid = cp.X == kXGlobal
                        ? dim3((unsigned)(cp.K * cp.dirs * nb), 1u, 1u)
                        : dim3((unsigned)cp.K, (unsigned)nb, (unsigned)cp.dirs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)cp.threads, 1, 1);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (started) {
    attr[na].id = cudaLaunchAttributeLaunchCompletionEvent;
    attr[na].val.launchCompletionEvent.event = started;
    attr[na].val.launchCompletionEvent.flags = 0;
    ++na;
  }
  if (cp.X != kXCluster) {
    // one band, or global-exchange bands: an ordinary launch (a CTA outside a
    // cluster is a cluster of one)
    *placed = true;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (started_used) *started_used = started != nullptr;
    return cudaLaunchKernelEx(&cfg, kern, p, ws, b0, cp);
  }
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)cp.K;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  // a cluster of K CTAs of this size must fit the GPU at all (asked once per
  // device and shape)
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, int, int, size_t>, int> fits;
  const auto key = std::make_tuple(dev, (const void *)kern, cp.K, cp.threads, bytes);
  int clusters = -1;
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = fits.find(key);
    if (it != fits.end()) clusters = it->second;
  }
  if (clusters < 0) {
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    fits[key] = clusters;
  }
  *placed = clusters >= 1;
  if (!*placed) return cudaSuccess;
  if (started_used) *started_used = started != nullptr;
  return cudaLaunchKernelEx(&cfg, kern, p, ws, b0, cp);
}

template <int ND>
cudaError_t launch_cluster(const Problem &p, const Workspace &ws, long long b0, long long nb,
                           bool with_beta, const ClusterPlan &cp, cudaStream_t stream,
                           bool *placed, cudaEvent_t started, bool *started_used) {
  return launch_cluster_g<ND, group_lanes(ND)>(p, ws, b0, nb, with_beta, cp, stream, placed,
                                               started, started_used);
}

// Launch the cluster variant; *placed is false (nothing launched) when a
// cluster of cp.K CTAs of this size does not fit the GPU.
cudaError_t launch_cluster_nd(const Problem &p, const Workspace &ws, long long b0, long long nb,
                              bool with_beta, const ClusterPlan &cp, cudaStream_t stream,
                              bool *placed, cudaEvent_t started, bool *started_used) {
  switch (p.n_dur) {
    case 1:
      return launch_cluster<1>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 2:
      return launch_cluster<2>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 3:
      return launch_cluster<3>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 4:
      return launch_cluster<4>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 5:
      return launch_cluster<5>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 6:
      return launch_cluster<6>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 7:
      return launch_cluster<7>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    case 8:
      return launch_cluster<8>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
    default:
      return launch_cluster<9>(p, ws, b0, nb, with_beta, cp, stream, placed, started,
                                started_used);
  }
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
    else L = -((double)ws.loglik[b].e * 0.69314718055994530942 + log((double)ws.loglik[b].s));
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


cudaError_t launch_lattice(const Problem &p_in, const Workspace &ws, long long b_begin,
                           long long b_end, bool with_beta, cudaStream_t stream,
                           cudaEvent_t started, bool *started_used) {
  Problem p = p_in;
  const long long limit = g_wait_limit.load();
  p.wait_limit = limit > 0 ? limit : kWaitLimitCycles;
  p.fault_utt = g_fault_utt.load();
  if (started_used) *started_used = false;
  if (b_end - b_begin > 65535) started = nullptr;
  // grid.y is at most 65535: launch in groups of utterances
  for (long long g0 = b_begin; g0 < b_end; g0 += 65535) {
    const long long nb = (b_end - g0 < 65535) ? b_end - g0 : 65535;
    bool done = false;
    // K bands per utterance: the preferred count, else more bands (fewer
    // rows, when a band needs too many threads or too much shared memory),
    // else fewer (when a cluster of K CTAs does not fit the GPU)
    if (p.gx_rows > 0) {
      // bands exchanging through global memory, as planned for the node
      // tables that cleared their boundary rows
      ClusterPlan cp;
      const bool alone = nb == p.B;  // the launch covers the whole batch
      if (cluster_plan(p, (int)((p.U1 + p.gx_rows - 1) / p.gx_rows), kXGlobal, &cp, alone) &&
          cp.Rc == p.gx_rows) {
        bool placed = false;
        const cudaError_t e = launch_cluster_nd(p, ws, g0, nb, with_beta, cp, stream, &placed,
                                                started, started_used);
        if (e != cudaSuccess) return e;
        done = placed;
      }
    }
    const int K0 = preferred_bands(p, nb);
    for (int step = 0; step < 2 * kMaxCluster && !done; ++step) {
      const int K = step < kMaxCluster - K0 + 1 ? K0 + step : K0 - (step - (kMaxCluster - K0));
      if (K < 1 || K > kMaxCluster) continue;
      ClusterPlan cp;
      if (!cluster_plan(p, K, kXCluster, &cp)) continue;
      bool placed = false;
      const cudaError_t e =
          launch_cluster_nd(p, ws, g0, nb, with_beta, cp, stream, &placed, started, started_used);
      if (e != cudaSuccess) return e;
      done = placed;
    }
    if (!done) {
      alpha_kernel<<<(unsigned)nb, lattice_threads(p), 0, stream>>>(p, ws, g0);
      if (with_beta) beta_kernel<<<(unsigned)nb, lattice_threads(p), 0, stream>>>(p, ws, g0);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_reduce(const Problem &p, const Workspace &ws, float *loss_out,
                          cudaStream_t stream) {
  reduce_kernel<<<1, 256, 0, stream>>>(p, ws, loss_out);
  return cudaGetLastError();
}

}  // namespace tdt

extern "C" int tdt_loss_set_lattice_bands(int bands) {
  if (bands < 0) bands = 0;
  return tdt::g_forced_bands.exchange(bands);
}

extern "C" int tdt_loss_set_lattice_exchange(int mode) {
  if (mode < 0 || mode > 2) mode = 0;
  return tdt::g_forced_exchange.exchange(mode);
}

extern "C" long long tdt_loss_test_set_halo_fault(long long utterance,
                                                  long long wait_limit_cycles) {
  tdt::g_wait_limit.store(wait_limit_cycles > 0 ? wait_limit_cycles : 0);
  return tdt::g_fault_utt.exchange(utterance >= 0 ? utterance : -1);
}
