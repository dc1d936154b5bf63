// tdt_api.cu -- the C ABI (include/tdt_loss.h): argument checks, scratch
// layout, and the order of the kernels.
//
// The batch is cut into up to kChunks groups of utterances, and the call
// forks from the caller's stream onto internal streams of three priorities:
//   * highest: one stream per chunk runs the alpha/beta lattice pass of
//     chunk c as soon as K1 of chunk c is done; the first of them then runs
//     the reduction once every chunk's lattice is done;
//   * middle: K1 node tables for chunk 0, 1, ... on two streams taken in
//     turn, each waiting for the end of the one before (with several
//     utterances a chunk, only K1 of chunk 1 does: the later ones follow the
//     pass before them on their own stream, so two run side by side).
//     K1 of chunk 1 also waits until every block of the lattice pass of
//     chunk 0 has started (a launch-completion event): a lattice block needs
//     an SM to itself, and once the next K1 pass has filled the GPU it was
//     measured to wait ~27 us for one.  Only the lattice of chunk 0 is on the
//     critical path; the later ones end long before their K4 passes start;
//   * lowest: K4 gradient of chunk c, once the lattice of chunk c is done,
//     on two streams taken in turn.
// The latency-bound lattice passes (a few SMs) run under the bandwidth-bound
// K1/K4 passes of other chunks instead of between them.  The block scheduler
// prefers pending blocks of higher-priority streams, so a K4 pass that is
// ready fills the SMs that the tail of the last K1 pass (or of the K4 pass
// before it) leaves idle instead of waiting for it to end.  The fork and the
// joins are CUDA events, so the whole call is stream-ordered (and
// capturable) on the caller's stream.
#include <math.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/tdt_loss.h"
#include "tdt_common.cuh"

namespace tdt {
namespace {

size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

bool make_layout(const int64_t sizes[4], int n_dur, Layout *L) {
  if (!sizes) return false;
  const long long B = sizes[0], T = sizes[1], U1 = sizes[2];
  if (B < 0 || T < 1 || U1 < 1 || n_dur < 1 || n_dur > kMaxDurations) return false;
  if (T + U1 > 65536) return false;
  const size_t ndiag = (size_t)B * (size_t)(T + U1 - 1) * (size_t)U1;
  const size_t nodes = (size_t)B * (size_t)T * (size_t)U1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L->arcw = take(ndiag * sizeof(LV) * (size_t)arc_record_len(n_dur));
  L->alpha = take(ndiag * sizeof(LV));
  L->beta = take(ndiag * sizeof(LV));
  L->lse_tok = take(nodes * 4);
  L->lse_dur = take(nodes * 4);
  L->frac = take(ndiag * 4 * (size_t)(2 + n_dur));
  L->loglik = take((size_t)B * sizeof(LV));
  L->scale = take((size_t)B * 4);
  L->usable = take((size_t)B * 4);
  L->ticket = take((size_t)B * 4);
  L->total = off > 0 ? off : 256;
  return true;
}

Workspace carve(const Layout &L, void *base) {
  char *c = static_cast<char *>(base);
  Workspace w;
  w.arcw = reinterpret_cast<LV *>(c + L.arcw);
  w.alpha = reinterpret_cast<LV *>(c + L.alpha);
  w.beta = reinterpret_cast<LV *>(c + L.beta);
  w.lse_tok = reinterpret_cast<float *>(c + L.lse_tok);
  w.lse_dur = reinterpret_cast<float *>(c + L.lse_dur);
  w.frac = reinterpret_cast<float *>(c + L.frac);
  w.loglik = reinterpret_cast<LV *>(c + L.loglik);
  w.scale = reinterpret_cast<float *>(c + L.scale);
  w.usable = reinterpret_cast<int *>(c + L.usable);
  w.ticket = reinterpret_cast<int *>(c + L.ticket);
  return w;
}

size_t elem_size(int dtype) { return dtype == TDT_DTYPE_F32 ? 4 : 2; }

// Host-side validation; fills the kernel parameter block.  No device access.
int validate(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
             const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
             const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
             const float *loss_out, const void *grad_out, Problem *p, bool need_loss,
             bool rnnt) {
  // plain RNN-T: no duration logits; the lattice has durations {0, 1}
  static const int32_t kRnntDurations[2] = {0, 1};
  if (rnnt) {
    durations = kRnntDurations;
    n_dur = 2;
  }
  const int n_dur_logits = rnnt ? 0 : n_dur;
  if (!sizes || !strides || !durations) return TDT_ERR_NULL_POINTER;
  // loss_out may be NULL only when it has no elements (empty batch, reduction none)
  if (need_loss && !loss_out && !(sizes[0] == 0 && reduction == TDT_REDUCTION_NONE))
    return TDT_ERR_NULL_POINTER;
  if (dtype != TDT_DTYPE_F32 && dtype != TDT_DTYPE_F16 && dtype != TDT_DTYPE_BF16)
    return TDT_ERR_BAD_DTYPE;
  if (n_dur < 1 || n_dur > kMaxDurations) return TDT_ERR_BAD_DURATIONS;
  const long long B = sizes[0], T = sizes[1], U1 = sizes[2], VD = sizes[3];
  if (B < 0 || T < 1 || U1 < 1 || VD <= n_dur_logits) return TDT_ERR_BAD_SIZES;
  if (T + U1 > 65536) return TDT_ERR_BAD_SIZES;
  if (B * T * U1 >= (1LL << 31)) return TDT_ERR_BAD_SIZES;
  if (B > 0 && (!logits || !logit_lens || !label_lens)) return TDT_ERR_NULL_POINTER;
  if (B > 0 && U1 > 1 && !labels) return TDT_ERR_NULL_POINTER;
  if (strides[3] != 1 || strides[0] < 0 || strides[1] < 0 || strides[2] < 0)
    return TDT_ERR_BAD_STRIDES;
  int max_dur = 0;
  for (int i = 0; i < n_dur; ++i) {
    if (durations[i] < 0 || durations[i] > kMaxDurationValue) return TDT_ERR_BAD_DURATIONS;
    for (int j = 0; j < i; ++j)
      if (durations[j] == durations[i]) return TDT_ERR_BAD_DURATIONS;
    if (durations[i] > max_dur) max_dur = durations[i];
  }
  const long long V = VD - n_dur_logits;
  if (blank < 0 || blank >= V) return TDT_ERR_BAD_BLANK;
  if (reduction < TDT_REDUCTION_NONE || reduction > TDT_REDUCTION_MEAN_VOLUME)
    return TDT_ERR_BAD_REDUCTION;
  if (!(fabs(sigma) <= 1024.0)) return TDT_ERR_BAD_SIGMA;
  const size_t es = elem_size(dtype);
  if (((uintptr_t)logits % es) != 0 || (grad_out && ((uintptr_t)grad_out % es) != 0) ||
      ((uintptr_t)loss_out % 4) != 0)
    return TDT_ERR_BAD_ALIGNMENT;
  // grad_out may overlap the logits only as the same contiguous tensor (the
  // gradient written in place over the logits, row by row)
  if (grad_out && B > 0) {
    const long long span = ((B - 1) * strides[0] + (T - 1) * strides[1] + (U1 - 1) * strides[2] +
                            VD) * (long long)es;
    const long long gspan = B * T * U1 * VD * (long long)es;
    const uintptr_t l0 = (uintptr_t)logits, g0 = (uintptr_t)grad_out;
    const bool overlap = g0 < l0 + (uintptr_t)span && l0 < g0 + (uintptr_t)gspan;
    const bool contiguous = strides[2] == VD && strides[1] == U1 * VD && strides[0] == T * U1 * VD;
    if (overlap && !(g0 == l0 && contiguous)) return TDT_ERR_BAD_ALIASING;
  }

  memset(p, 0, sizeof(*p));
  p->logits = logits;
  p->B = B; p->T = T; p->U1 = U1; p->VD = VD; p->V = V; p->D = n_dur_logits;
  p->s0 = strides[0]; p->s1 = strides[1]; p->s2 = strides[2];
  p->labels = reinterpret_cast<const long long *>(labels);
  p->logit_lens = reinterpret_cast<const long long *>(logit_lens);
  p->label_lens = reinterpret_cast<const long long *>(label_lens);
  for (int i = 0; i < n_dur; ++i) p->dur[i] = durations[i];
  p->n_dur = n_dur;
  p->max_dur = max_dur;
  p->blank = blank;
  p->reduction = reduction;
  p->sigma_fx = (fx_t)llround(sigma * kFxOne);
  p->n_diag = T + U1 - 1;
  p->rec_len = arc_record_len(n_dur);
  p->rnnt = rnnt ? 1 : 0;
  fast_div_setup(T, &p->divT_m, &p->divT_s);
  fast_div_setup(U1, &p->divU1_m, &p->divU1_s);
  p->gx_rows = 0;
  return TDT_OK;
}

namespace {

// ---- optional per-kernel timing (benchmarks) --------------------------------
// Each call records a reference event on the caller's stream before its first
// kernel; every timed launch records an event pair on its own stream.  A
// kernel's busy window in a call runs from the start of its first launch to
// the end of its last one (launches of one kernel may overlap on several
// streams), measured from the call's reference event.
struct Timing {
  std::mutex mu;
  bool on = false;
  struct Pending { int id; long long call; cudaEvent_t a, b; };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> call_ref;  // reference event of call k (k = index)
  std::vector<cudaEvent_t> pool;
  double ms[TDT_KERNEL_COUNT] = {0};
  double span[TDT_KERNEL_COUNT] = {0};
  long long count[TDT_KERNEL_COUNT] = {0};
};
Timing &timing() {
  static Timing t;
  return t;
}
cudaEvent_t take_event(Timing &t) {
  if (!t.pool.empty()) {
    cudaEvent_t e = t.pool.back();
    t.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Start of a call: its reference event, when timing is on.
void begin_timed_call(cudaStream_t stream) {
  Timing &t = timing();
  std::lock_guard<std::mutex> g(t.mu);
  if (!t.on) return;
  cudaEvent_t e = take_event(t);
  cudaEventRecord(e, stream);
  t.call_ref.push_back(e);
}

// Launch one kernel through `fn`, bracketed by events when timing is on.
template <class F>
cudaError_t timed(int id, cudaStream_t stream, F fn) {
  Timing &t = timing();
  bool on;
  long long call;
  {
    std::lock_guard<std::mutex> g(t.mu);
    on = t.on && !t.call_ref.empty();
    call = (long long)t.call_ref.size() - 1;
  }
  if (!on) return fn();
  cudaEvent_t a, b;
  {
    std::lock_guard<std::mutex> g(t.mu);
    a = take_event(t);
    b = take_event(t);
  }
  cudaEventRecord(a, stream);
  cudaError_t e = fn();
  cudaEventRecord(b, stream);
  std::lock_guard<std::mutex> g(t.mu);
  t.pending.push_back({id, call, a, b});
  return e;
}

// ---- per-device internal stream and events -----------------------------------
constexpr int kChunks = 4;
constexpr long long kSerialBytes = 8ll << 20;  // below: one stream, no chunks

struct DeviceRes {
  bool ready = false;
  cudaStream_t side[kChunks] = {};  // highest priority, one per chunk's lattice pass
  cudaStream_t tables[2] = {};      // middle priority: the K1 passes, in turn
  cudaStream_t grad[2] = {};        // lowest priority: the K4 passes, in turn
  cudaEvent_t fork = nullptr, join = nullptr, tables_end[2] = {}, grad_end[2] = {};
  cudaEvent_t tables_done[kChunks] = {}, lattice_done[kChunks] = {}, started[kChunks] = {};
  std::mutex mu;                // one call at a time enqueues on these events
};

DeviceRes *device_res(int dev) {
  static std::mutex mu;
  static std::vector<DeviceRes *> all;
  std::lock_guard<std::mutex> g(mu);
  if ((int)all.size() <= dev) all.resize(dev + 1, nullptr);
  if (!all[dev]) all[dev] = new DeviceRes();  // lives until process exit
  DeviceRes *r = all[dev];
  if (!r->ready) {
    int lo = 0, hi = 0;  // least and greatest priority (greatest = smallest number)
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) return nullptr;
    const int mid = hi < lo ? hi + 1 : lo;
    for (int c = 0; c < kChunks; ++c)
      if (cudaStreamCreateWithPriority(&r->side[c], cudaStreamNonBlocking, hi) != cudaSuccess)
        return nullptr;
    for (int i = 0; i < 2; ++i)
      if (cudaStreamCreateWithPriority(&r->tables[i], cudaStreamNonBlocking, mid) != cudaSuccess ||
          cudaStreamCreateWithPriority(&r->grad[i], cudaStreamNonBlocking, lo) != cudaSuccess)
        return nullptr;
    bool ok = true;
    for (cudaEvent_t *e : {&r->fork, &r->join, &r->tables_end[0], &r->tables_end[1],
                           &r->grad_end[0], &r->grad_end[1]})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; c < kChunks && ok; ++c)
      ok = cudaEventCreateWithFlags(&r->tables_done[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&r->lattice_done[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&r->started[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    r->ready = true;
  }
  return r;
}

// One loss (+ gradient) call.  coeffs: also run beta and the arc fractions
// (always when grad_out is given; the forward half of the split API keeps
// them for the backward half).  gscale: upstream gradient of the
// loss (device, NULL = 1).
int run(const Problem &p, int dtype, const Workspace &ws, float *loss_out, void *grad_out,
        const float *gscale, bool coeffs, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TDT_ERR_CUDA;
  DeviceRes *res = device_res(dev);
  if (!res) return TDT_ERR_CUDA;
  std::lock_guard<std::mutex> g(res->mu);
  begin_timed_call(stream);
  const bool with_grad = grad_out != nullptr;
  coeffs = coeffs || with_grad;
  const long long rows_per_utt = p.T * p.U1;
#define TDT_TRY(x) \
  do {             \
    if ((x) != cudaSuccess) return TDT_ERR_CUDA; \
  } while (0)
  // Small problems (logits below kSerialBytes): launch latency, not
  // bandwidth, sets the time, so the kernels run one after another on the
  // caller's stream with no fork, join or chunking.
  const long long logit_bytes = p.B * rows_per_utt * p.VD * (dtype == kF32 ? 4 : 2);
  if (logit_bytes < kSerialBytes) {
    const long long rows = p.B * rows_per_utt;
    Problem ps = p;
    ps.gx_rows = lattice_global_rows(p, p.B);
    TDT_TRY(timed(TDT_KERNEL_TABLES, stream,
                  [&] { return launch_node_tables(ps, dtype, ws, 0, rows, stream); }));
    TDT_TRY(timed(TDT_KERNEL_LATTICE, stream,
                  [&] { return launch_lattice(ps, ws, 0, p.B, coeffs, stream); }));
    TDT_TRY(timed(TDT_KERNEL_REDUCE, stream, [&] { return launch_reduce(p, ws, loss_out, stream); }));
    if (with_grad)
      TDT_TRY(timed(TDT_KERNEL_GRAD, stream, [&] {
        return launch_grad(p, dtype, ws, grad_out, gscale, 0, rows, stream);
      }));
    return TDT_OK;
  }
  const int nchunk = (int)(p.B < kChunks ? (p.B > 0 ? p.B : 1) : kChunks);
  auto b_lo = [&](int c) { return p.B * c / nchunk; };
  TDT_TRY(cudaEventRecord(res->fork, stream));
  for (int c = 0; c < nchunk; ++c) TDT_TRY(cudaStreamWaitEvent(res->side[c], res->fork, 0));
  const int nts = nchunk < 2 ? nchunk : 2;
  bool started_used = false;
  for (int i = 0; i < nts; ++i) TDT_TRY(cudaStreamWaitEvent(res->tables[i], res->fork, 0));
  for (int c = 0; c < nchunk; ++c) {
    const long long b0 = b_lo(c), b1 = b_lo(c + 1);
    cudaStream_t side = res->side[c], ts = res->tables[c & 1];
    // K1(c) waits for K1(c - 1) (the utterance order of the lattices); for
    // chunks of several utterances only K1(1) does, and K1(2), K1(3) follow
    // the pass before them on their own stream, so two run side by side
    // (large_batch, four utterances a chunk: 1.457 vs 1.480 ms per step;
    // with one utterance a chunk the overlapping passes were slower)
    if (c == 1 || (c > 1 && b1 - b0 < 2))
      TDT_TRY(cudaStreamWaitEvent(ts, res->tables_done[c - 1], 0));
    if (c == 1 && started_used) TDT_TRY(cudaStreamWaitEvent(ts, res->started[0], 0));
    // the band plan of this chunk's lattice: its node tables clear the
    // boundary rows that the bands exchange through global memory
    Problem pc = p;
    pc.gx_rows = lattice_global_rows(p, b1 - b0);
    TDT_TRY(timed(TDT_KERNEL_TABLES, ts, [&] {
      return launch_node_tables(pc, dtype, ws, b0 * rows_per_utt, b1 * rows_per_utt, ts);
    }));
    TDT_TRY(cudaEventRecord(res->tables_done[c], ts));
    TDT_TRY(cudaStreamWaitEvent(side, res->tables_done[c], 0));
    started_used = false;
    TDT_TRY(timed(TDT_KERNEL_LATTICE, side, [&] {
      return launch_lattice(pc, ws, b0, b1, coeffs, side,
                            c == 0 && nchunk > 1 ? res->started[0] : nullptr, &started_used);
    }));
    TDT_TRY(cudaEventRecord(res->lattice_done[c], side));
  }
  for (int i = 0; i < nts; ++i) TDT_TRY(cudaEventRecord(res->tables_end[i], res->tables[i]));
  // the reduction needs every chunk's log-likelihood; it joins all side streams
  cudaStream_t side0 = res->side[0];
  for (int c = 1; c < nchunk; ++c) TDT_TRY(cudaStreamWaitEvent(side0, res->lattice_done[c], 0));
  TDT_TRY(timed(TDT_KERNEL_REDUCE, side0, [&] { return launch_reduce(p, ws, loss_out, side0); }));
  TDT_TRY(cudaEventRecord(res->join, side0));
  for (int i = 0; i < nts; ++i) TDT_TRY(cudaStreamWaitEvent(stream, res->tables_end[i], 0));
  TDT_TRY(cudaStreamWaitEvent(stream, res->join, 0));
  if (with_grad) {
    const int ngs = nchunk < 2 ? nchunk : 2;
    for (int i = 0; i < ngs; ++i) TDT_TRY(cudaStreamWaitEvent(res->grad[i], res->fork, 0));
    for (int c = 0; c < nchunk; ++c) {
      const long long b0 = b_lo(c), b1 = b_lo(c + 1);
      cudaStream_t gs = res->grad[c & 1];
      TDT_TRY(cudaStreamWaitEvent(gs, res->lattice_done[c], 0));
      TDT_TRY(timed(TDT_KERNEL_GRAD, gs, [&] {
        return launch_grad(p, dtype, ws, grad_out, gscale, b0 * rows_per_utt, b1 * rows_per_utt,
                           gs);
      }));
    }
    for (int i = 0; i < ngs; ++i) {
      TDT_TRY(cudaEventRecord(res->grad_end[i], res->grad[i]));
      TDT_TRY(cudaStreamWaitEvent(stream, res->grad_end[i], 0));
    }
  }
#undef TDT_TRY
  return TDT_OK;
}

// The backward half of the split API: the gradient pass over every row.
int run_bwd(const Problem &p, int dtype, const Workspace &ws, void *grad_out, const float *gscale,
            cudaStream_t stream) {
  if (p.B == 0) return TDT_OK;
  begin_timed_call(stream);
  if (timed(TDT_KERNEL_GRAD, stream, [&] {
        return launch_grad(p, dtype, ws, grad_out, gscale, 0, p.B * p.T * p.U1, stream);
      }) != cudaSuccess)
    return TDT_ERR_CUDA;
  return TDT_OK;
}

// Checks shared by the entry points that take caller-owned scratch.
int check_workspace(const int64_t sizes[4], int n_dur, const void *workspace,
                    size_t workspace_bytes, Workspace *ws) {
  Layout L;
  if (!make_layout(sizes, n_dur, &L)) return TDT_ERR_BAD_SIZES;
  if (!workspace) return TDT_ERR_NULL_POINTER;
  if (workspace_bytes < L.total) return TDT_ERR_WORKSPACE_TOO_SMALL;
  if (((uintptr_t)workspace % 256) != 0) return TDT_ERR_BAD_ALIGNMENT;
  *ws = carve(L, const_cast<void *>(workspace));
  return TDT_OK;
}

}  // namespace
}  // namespace tdt

extern "C" {

size_t tdt_loss_workspace_size(const int64_t sizes[4], int n_dur) {
  tdt::Layout L;
  if (!tdt::make_layout(sizes, n_dur, &L)) return 0;
  return L.total;
}

int tdt_loss_fwd_bwd_ws(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                        int dtype, const int64_t *labels, const int64_t *logit_lens,
                        const int64_t *label_lens, const int32_t *durations, int n_dur,
                        int blank, double sigma, int reduction, float *loss_out, void *grad_out,
                        void *workspace, size_t workspace_bytes, void *stream) {
  tdt::Problem p;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens,
                         durations, n_dur, blank, sigma, reduction, loss_out, grad_out, &p, true);
  if (rc != TDT_OK) return rc;
  tdt::Workspace ws;
  rc = tdt::check_workspace(sizes, n_dur, workspace, workspace_bytes, &ws);
  if (rc != TDT_OK) return rc;
  return tdt::run(p, dtype, ws, loss_out, grad_out, nullptr, false,
                  static_cast<cudaStream_t>(stream));
}

int tdt_loss_fwd(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
                 const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
                 const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
                 float *loss_out, void *workspace, size_t workspace_bytes, void *stream) {
  tdt::Problem p;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens,
                         durations, n_dur, blank, sigma, reduction, loss_out, nullptr, &p, true);
  if (rc != TDT_OK) return rc;
  tdt::Workspace ws;
  rc = tdt::check_workspace(sizes, n_dur, workspace, workspace_bytes, &ws);
  if (rc != TDT_OK) return rc;
  return tdt::run(p, dtype, ws, loss_out, nullptr, nullptr, true,
                  static_cast<cudaStream_t>(stream));
}

int tdt_loss_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
                 const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
                 const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
                 const float *grad_loss, void *grad_out, const void *workspace,
                 size_t workspace_bytes, void *stream) {
  tdt::Problem p;
  if (!grad_out) return TDT_ERR_NULL_POINTER;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens,
                         durations, n_dur, blank, sigma, reduction, nullptr, grad_out, &p, false);
  if (rc != TDT_OK) return rc;
  if (((uintptr_t)grad_loss % 4) != 0) return TDT_ERR_BAD_ALIGNMENT;
  tdt::Workspace ws;
  rc = tdt::check_workspace(sizes, n_dur, workspace, workspace_bytes, &ws);
  if (rc != TDT_OK) return rc;
  return tdt::run_bwd(p, dtype, ws, grad_out, grad_loss, static_cast<cudaStream_t>(stream));
}

int tdt_loss_fwd_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                     int dtype, const int64_t *labels, const int64_t *logit_lens,
                     const int64_t *label_lens, const int32_t *durations, int n_dur, int blank,
                     double sigma, int reduction, float *loss_out, void *grad_out,
                     void *stream) {
  tdt::Problem p;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens,
                         durations, n_dur, blank, sigma, reduction, loss_out, grad_out, &p, true);
  if (rc != TDT_OK) return rc;
  tdt::Layout L;
  if (!tdt::make_layout(sizes, n_dur, &L)) return TDT_ERR_BAD_SIZES;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *ws_ptr = nullptr;
  if (cudaMallocAsync(&ws_ptr, L.total, s) != cudaSuccess) return TDT_ERR_CUDA;
  tdt::Workspace ws = tdt::carve(L, ws_ptr);
  rc = tdt::run(p, dtype, ws, loss_out, grad_out, nullptr, false, s);
  if (cudaFreeAsync(ws_ptr, s) != cudaSuccess && rc == TDT_OK) rc = TDT_ERR_CUDA;
  return rc;
}

int tdt_rnnt_loss_fwd_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                          int dtype, const int64_t *labels, const int64_t *logit_lens,
                          const int64_t *label_lens, int blank, double sigma, int reduction,
                          float *loss_out, void *grad_out, void *stream) {
  tdt::Problem p;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens, nullptr,
                         0, blank, sigma, reduction, loss_out, grad_out, &p, true, true);
  if (rc != TDT_OK) return rc;
  tdt::Layout L;
  if (!tdt::make_layout(sizes, p.n_dur, &L)) return TDT_ERR_BAD_SIZES;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *ws_ptr = nullptr;
  if (cudaMallocAsync(&ws_ptr, L.total, s) != cudaSuccess) return TDT_ERR_CUDA;
  tdt::Workspace ws = tdt::carve(L, ws_ptr);
  rc = tdt::run(p, dtype, ws, loss_out, grad_out, nullptr, false, s);
  if (cudaFreeAsync(ws_ptr, s) != cudaSuccess && rc == TDT_OK) rc = TDT_ERR_CUDA;
  return rc;
}

const char *tdt_status_string(int status) {
  switch (status) {
    case TDT_OK: return "ok";
    case TDT_ERR_NULL_POINTER: return "a required pointer is NULL";
    case TDT_ERR_BAD_SIZES: return "invalid sizes (B>=0, T>=1, U+1>=1, V+D>n_dur, T+U+1<=65536)";
    case TDT_ERR_BAD_STRIDES: return "invalid strides (strides[3] must be 1, others >= 0)";
    case TDT_ERR_BAD_DTYPE: return "unknown dtype";
    case TDT_ERR_BAD_DURATIONS:
      return "invalid durations (1..32 distinct values in [0, 255])";
    case TDT_ERR_BAD_BLANK: return "blank outside [0, V)";
    case TDT_ERR_BAD_REDUCTION: return "unknown reduction";
    case TDT_ERR_BAD_SIGMA: return "sigma must be finite with |sigma| <= 1024";
    case TDT_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than tdt_loss_workspace_size";
    case TDT_ERR_CUDA: return "a CUDA call failed";
    case TDT_ERR_BAD_ALIGNMENT: return "a pointer is not aligned to its element size";
    case TDT_ERR_BAD_ALIASING:
      return "grad_out overlaps the logits other than as the same contiguous tensor";
    case TDT_ERR_NOALLOC_TOO_LARGE:
      return "problem needs more scratch than the fixed array of tdt_loss_fwd_bwd_noalloc "
             "(TDT_NOALLOC_MAX_WORKSPACE_BYTES); use tdt_loss_fwd_bwd or tdt_loss_fwd_bwd_ws";
    default: return "unknown status";
  }
}

int tdt_loss_version(void) { return TDT_LOSS_VERSION; }

void tdt_loss_timing_enable(int on) {
  tdt::Timing &t = tdt::timing();
  std::lock_guard<std::mutex> g(t.mu);
  t.on = on != 0;
}

int tdt_loss_timing_read(double *ms_out, int64_t *count_out, double *span_ms_out, int n,
                         int reset) {
  tdt::Timing &t = tdt::timing();
  std::lock_guard<std::mutex> g(t.mu);
  int rc = 0;
  // per call and kernel: earliest start and latest end after the reference
  std::vector<float> lo(t.call_ref.size() * TDT_KERNEL_COUNT, 1e30f);
  std::vector<float> hi(t.call_ref.size() * TDT_KERNEL_COUNT, -1e30f);
  for (auto &pe : t.pending) {
    float ms = 0.0f, s0 = 0.0f, s1 = 0.0f;
    const cudaEvent_t ref = t.call_ref[pe.call];
    if (cudaEventSynchronize(pe.b) != cudaSuccess ||
        cudaEventElapsedTime(&ms, pe.a, pe.b) != cudaSuccess ||
        cudaEventElapsedTime(&s0, ref, pe.a) != cudaSuccess ||
        cudaEventElapsedTime(&s1, ref, pe.b) != cudaSuccess)
      rc = TDT_ERR_CUDA;
    t.ms[pe.id] += ms;
    t.count[pe.id] += 1;
    const size_t k = (size_t)pe.call * TDT_KERNEL_COUNT + pe.id;
    if (s0 < lo[k]) lo[k] = s0;
    if (s1 > hi[k]) hi[k] = s1;
    t.pool.push_back(pe.a);
    t.pool.push_back(pe.b);
  }
  for (size_t k = 0; k < lo.size(); ++k)
    if (hi[k] >= lo[k]) t.span[k % TDT_KERNEL_COUNT] += hi[k] - lo[k];
  t.pending.clear();
  for (cudaEvent_t e : t.call_ref) t.pool.push_back(e);
  t.call_ref.clear();
  if (n > TDT_KERNEL_COUNT) n = TDT_KERNEL_COUNT;
  for (int i = 0; i < n; ++i) {
    if (ms_out) ms_out[i] = t.ms[i];
    if (count_out) count_out[i] = t.count[i];
    if (span_ms_out) span_ms_out[i] = t.span[i];
  }
  if (reset)
    for (int i = 0; i < TDT_KERNEL_COUNT; ++i) {
      t.ms[i] = 0.0;
      t.span[i] = 0.0;
      t.count[i] = 0;
    }
  return rc != 0 ? rc : (n < 0 ? 0 : n);
}

}  // extern "C"
