/*
 * tdt_loss.h -- C ABI of the GB300 (sm_103a) Token-and-Duration Transducer
 * (TDT) loss: forward and backward in one call, or split in two for autograd.
 *
 * The operation ("tdt-loss: add TDT loss kernel", kernels-community PR
 * #882, list "What's in it"):
 *   - a log-softmax over the vocabulary at every lattice node, and one over
 *     the duration logits;
 *   - alpha/beta passes over the (t,u) lattice, no limit of 1024 labels;
 *     here in the probability domain with an exact int32 exponent beside
 *     each fp32 mantissa, so no value underflows however long the lattice;
 *   - one fused pass that writes the gradient w.r.t. the token and the
 *     duration logits;
 *   - fp32/fp16/bf16 logits read directly, including a slice
 *     logits[..., :V+D] of a wider tensor, without a copy;
 *   - the reductions mean_volume, mean_batch, mean, sum, none.
 * sigma, the logit under-normalisation, is a loss parameter ("Add TDT loss
 * kernel", transformers PR #46048, review: "test for sigma != 0").
 *
 * Lattice (published TDT, Xu et al. 2023): node (t,u), t < T_b, u <= U_b;
 * blank arc (t,u)->(t+d,u) for d > 0; label arc (t,u)->(t+d,u+1) for every
 * d incl. 0, landing before frame T_b; a path ends with a blank arc from
 * (t,U_b) that lands exactly on T_b.  Arc weight = token log-prob - sigma +
 * duration log-prob.  L_b = -log(sum over paths of exp(path weight)).
 *
 * Conventions common to every entry point
 *   logits      device, [B, T, U+1, V+D] of `dtype`, addressed with the
 *               element strides `strides` (strides[3] must be 1; the other
 *               strides are free, e.g. a slice of a [..., W] tensor with
 *               W > V+D).  Token logits are [..., 0:V) with `blank` inside,
 *               duration logits [..., V:V+D), D = n_dur.
 *   sizes       host, {B, T, U+1, V+D}; B >= 0, T >= 1, U+1 >= 1,
 *               V+D > n_dur, T + U + 1 <= 65536, B * T * (U+1) < 2^31.
 *   labels      device int64 [B, U] contiguous (U = sizes[2]-1); entries at
 *               u >= label_lens[b] are ignored (-100 padding).  May be NULL
 *               when U = 0.
 *   logit_lens  device int64 [B]: T_b.     label_lens: device int64 [B]: U_b.
 *   durations   host int32 [n_dur], distinct, 0 <= d <= 255; 1 <= n_dur <= 32.
 *   blank       index of blank in [0, V).
 *   sigma       under-normalisation, |sigma| <= 1024.
 *   reduction   one of TDT_REDUCTION_*.
 *   loss_out    device float32: [B] for TDT_REDUCTION_NONE, else [1]
 *               (NULL allowed only for B = 0 with TDT_REDUCTION_NONE).
 *   grad_out    device, contiguous [B, T, U+1, V+D] of `dtype`; the
 *               gradient of the reduced loss for an upstream gradient of 1
 *               (of sum_b L_b for NONE).  NULL computes the loss only.
 *               Rows outside an utterance's lattice are written as 0.
 *               grad_out may be the logits pointer itself when the logits
 *               are contiguous: the gradient then replaces the logits, so
 *               no second [B,T,U+1,V+D] buffer is needed (a memory-lean
 *               option; the pages report a lower training peak memory with
 *               the fused kernel, "Fine-tune check": 33.6 -> 21.8 GiB).
 *               Any other overlap of grad_out with the logits is rejected
 *               with TDT_ERR_BAD_ALIASING.
 *   stream      a cudaStream_t (NULL: the legacy default stream).
 * Memory: the caller owns every pointer; the library never frees them.
 * Calls are asynchronous on `stream`: results are valid once the stream
 * reaches them.  No call synchronises the device.
 * Errors: a negative TDT_ERR_* status is returned before anything is
 * enqueued when an argument is invalid.  Problems that only the device can
 * see never trap: an utterance with T_b < 1, T_b > T, U_b < 0, U_b > U, or a
 * used label outside [0,V) or equal to blank gets a NaN loss and zero
 * gradient rows; an utterance with no complete path gets +inf and zero rows.
 * Log-probabilities below -4096 are clamped to -4096 (exp(-4096) is far
 * below the float64 range).
 */
#ifndef TDT_LOSS_H
#define TDT_LOSS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TDT_LOSS_VERSION 1

/* element type of logits and grad_out */
#define TDT_DTYPE_F32 0
#define TDT_DTYPE_F16 1
#define TDT_DTYPE_BF16 2

/* reductions ("supports all reductions: mean_volume, mean_batch, mean, sum, none") */
#define TDT_REDUCTION_NONE 0        /* loss_out[b] = L_b                          */
#define TDT_REDUCTION_SUM 1         /* sum_b L_b                                  */
#define TDT_REDUCTION_MEAN 2        /* (1/B) sum_b L_b / U_b                      */
#define TDT_REDUCTION_MEAN_BATCH 3  /* (1/B) sum_b L_b                            */
#define TDT_REDUCTION_MEAN_VOLUME 4 /* sum_b L_b / sum_b U_b                      */

/* status codes */
#define TDT_OK 0
#define TDT_ERR_NULL_POINTER (-1)
#define TDT_ERR_BAD_SIZES (-2)
#define TDT_ERR_BAD_STRIDES (-3)
#define TDT_ERR_BAD_DTYPE (-4)
#define TDT_ERR_BAD_DURATIONS (-5)
#define TDT_ERR_BAD_BLANK (-6)
#define TDT_ERR_BAD_REDUCTION (-7)
#define TDT_ERR_BAD_SIGMA (-8)
#define TDT_ERR_WORKSPACE_TOO_SMALL (-9)
#define TDT_ERR_CUDA (-10)
#define TDT_ERR_BAD_ALIGNMENT (-11)
#define TDT_ERR_NOALLOC_TOO_LARGE (-12)
#define TDT_ERR_BAD_ALIASING (-13)

/*
 * Loss and gradient in one call.  Internal scratch (per-node tables, alpha,
 * beta; tdt_loss_workspace_size bytes) is taken from the stream-ordered
 * allocator (cudaMallocAsync / cudaFreeAsync on `stream`).
 * When the logits reach 8 MiB, the work is spread over a few internal
 * streams of the current device (created once per device, of several
 * priorities) that fork from `stream` and join back to it through events,
 * so the call stays ordered on `stream` and can be captured into a CUDA
 * graph; smaller problems run their kernels one after another on `stream`.  Calls on one device are enqueued one at a
 * time (an internal lock); their GPU work is ordered by the internal streams
 * and events.
 * Returns TDT_OK or a TDT_ERR_* status.
 */
int tdt_loss_fwd_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                     int dtype, const int64_t *labels, const int64_t *logit_lens,
                     const int64_t *label_lens, const int32_t *durations, int n_dur, int blank,
                     double sigma, int reduction, float *loss_out, void *grad_out, void *stream);

/*
 * Plain RNN-T loss (no duration head) and its gradient, on the same kernels:
 * "Add TDT loss kernel" (transformers PR #46048), commit list, notes that
 * torchaudio's rnnt_loss does not train the duration head -- this is that
 * loss.  Lattice: blank arc (t,u)->(t+1,u), label arc (t,u)->(t,u+1), a path
 * ends with the blank arc from (T_b-1, U_b); arc weight = token log-prob -
 * sigma (sigma = 0: the textbook loss).
 *   logits  [B, T, U+1, V] (no duration logits), sizes = {B, T, U+1, V};
 *   every other argument as for tdt_loss_fwd_bwd (no durations);
 *   grad_out contiguous [B, T, U+1, V] or NULL; may be the logits (in place).
 */
int tdt_rnnt_loss_fwd_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                          int dtype, const int64_t *labels, const int64_t *logit_lens,
                          const int64_t *label_lens, int blank, double sigma, int reduction,
                          float *loss_out, void *grad_out, void *stream);

/*
 * Greedy TDT decoding over precomputed joint outputs ("Add TDT loss kernel",
 * transformers PR #46048, commit list: greedy TDT decoding with per-token
 * timestamps and token durations, and a max_symbols_per_step guard).  With
 * the joint output z[b,t,u,:] given for every frame t and decoder state u
 * (u tokens emitted), utterance b is decoded by the walk: start at (0,0);
 * at (t,u) take k = first argmax of z[0:V) and d = durations[first argmax of
 * z[V:V+D)]; a token k != blank is emitted with frame t and duration d and
 * u advances (decoding stops when row u would exceed U); a blank, or any
 * token once max_symbols tokens were emitted at this frame, moves at least
 * one frame; otherwise t advances by d; decoding stops at t >= T_b.
 *   logits, sizes, strides, dtype, logit_lens, durations, n_dur, blank:
 *             as for tdt_loss_fwd_bwd (no labels);
 *   max_symbols  >= 1;
 *   n_out          device int32 [B]: tokens decoded for each utterance;
 *   tokens_out, frames_out, durations_out  device int32 [B, U+1]: token,
 *             frame of emission and predicted duration, -1 past n_out[b].
 * An utterance with T_b < 1 or T_b > T decodes to nothing.  Ties go to the
 * smallest index; logits are expected to be finite.
 */
int tdt_greedy_decode(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                      int dtype, const int64_t *logit_lens, const int32_t *durations, int n_dur,
                      int blank, int max_symbols, int32_t *n_out, int32_t *tokens_out,
                      int32_t *frames_out, int32_t *durations_out, void *stream);

/*
 * Bytes of device scratch that tdt_loss_fwd_bwd_ws needs for these sizes
 * (0 for invalid arguments).  The value depends only on sizes and n_dur.
 */
size_t tdt_loss_workspace_size(const int64_t sizes[4], int n_dur);

/*
 * Same as tdt_loss_fwd_bwd, with caller-owned scratch: `workspace` is a
 * device pointer, 256-byte aligned, of at least workspace_bytes >=
 * tdt_loss_workspace_size(sizes, n_dur) bytes, not used by anything else
 * until the stream has passed this call.  Nothing is allocated.
 */
int tdt_loss_fwd_bwd_ws(const void *logits, const int64_t sizes[4], const int64_t strides[4],
                        int dtype, const int64_t *labels, const int64_t *logit_lens,
                        const int64_t *label_lens, const int32_t *durations, int n_dur,
                        int blank, double sigma, int reduction, float *loss_out,
                        void *grad_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The loss and its gradient in two calls, for autograd: the forward call
 * computes the loss and keeps in `workspace` everything the gradient needs;
 * the backward call, made later with the same arguments and the same
 * workspace, writes the gradient for an upstream gradient `grad_loss`.
 * The pages' layer supports backward and, through fake implementations of
 * its ops, torch.compile ("Add TDT loss kernel", transformers PR #46048,
 * review thread on the kernel mapping).
 *
 * tdt_loss_fwd: node tables, alpha, beta, the arc fractions and the
 *   reduction into loss_out.  workspace as for tdt_loss_fwd_bwd_ws; its
 *   contents must stay untouched until tdt_loss_bwd has run.
 */
int tdt_loss_fwd(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
                 const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
                 const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
                 float *loss_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * tdt_loss_bwd: the gradient pass only.  grad_loss is the device float32
 *   upstream gradient of loss_out ([B] for TDT_REDUCTION_NONE, else [1]) or
 *   NULL for 1; grad_out[b,...] = grad_loss[b or 0] * dL/dz.  Every other
 *   argument must equal the tdt_loss_fwd call's, and that call must come
 *   before this one in stream order.  grad_out is required (may be the
 *   logits themselves, see grad_out above).
 */
int tdt_loss_bwd(const void *logits, const int64_t sizes[4], const int64_t strides[4], int dtype,
                 const int64_t *labels, const int64_t *logit_lens, const int64_t *label_lens,
                 const int32_t *durations, int n_dur, int blank, double sigma, int reduction,
                 const float *grad_loss, void *grad_out, const void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Same loss and gradient as tdt_loss_fwd_bwd for callers that cannot
 * allocate device memory (the pages have no counterpart: this is an addition
 * of this library).  Some callers may not call cudaMalloc or any allocator:
 * code running while another component owns the device memory pool, or
 * runtimes that reserve all memory at start-up and treat a later
 * allocation as an error.  This entry point allocates nothing: its scratch
 * is a fixed device array of TDT_NOALLOC_MAX_WORKSPACE_BYTES inside the
 * library, held on every device that loads the library until the process
 * exits.  The caller still passes every input and output buffer.
 *   - Problems whose tdt_loss_workspace_size exceeds the array are rejected
 *     with TDT_ERR_NOALLOC_TOO_LARGE before anything is enqueued.
 *   - All calls on a device share the array: calls whose GPU work overlaps
 *     (other streams, unordered host threads) race.  Order them on one
 *     stream.  No entry of the array has to start at zero.
 *   - The first call in each CUDA context looks up the array's device
 *     address with that context current and keeps it under the context's
 *     unique id: the first call on a device, and again the first call after
 *     cudaDeviceReset or with another context current.  Make that first
 *     call before any stream capture.
 *   - The kernels run one after another on `stream`; no internal stream or
 *     event is created.
 */
#define TDT_NOALLOC_MAX_WORKSPACE_BYTES (64u * 1024u * 1024u)
int tdt_loss_fwd_bwd_noalloc(const void *logits, const int64_t sizes[4],
                             const int64_t strides[4], int dtype, const int64_t *labels,
                             const int64_t *logit_lens, const int64_t *label_lens,
                             const int32_t *durations, int n_dur, int blank, double sigma,
                             int reduction, float *loss_out, void *grad_out, void *stream);

/*
 * Benchmark support (not needed for correctness).  Kernel ids: node tables,
 * lattice (alpha and beta), reduction, gradient.
 */
#define TDT_KERNEL_TABLES 0
#define TDT_KERNEL_LATTICE 1
#define TDT_KERNEL_REDUCE 2
#define TDT_KERNEL_GRAD 3
#define TDT_KERNEL_COUNT 4

/*
 * on != 0: every later call records a CUDA event pair around each of its
 * kernels, on the stream that kernel is launched on; on == 0 stops it.
 * Process-wide; not meant for stream capture.
 */
void tdt_loss_timing_enable(int on);

/*
 * Per kernel id, for the first n ids, since the last reset: the sum of the
 * recorded launch durations in milliseconds (ms_out), the number of launches
 * (count_out), and the sum over calls of the kernel's busy window in the
 * call (span_ms_out): from the start of its first launch to the end of its
 * last launch in that call.  Launches of one kernel run on several streams
 * and may overlap, so span_ms_out can be less than ms_out.  Any output may
 * be NULL.  Blocks until the recorded events have completed.  reset != 0
 * clears the sums afterwards.  Returns the number of ids written or
 * TDT_ERR_CUDA.  Timing assumes one host thread making calls.
 */
int tdt_loss_timing_read(double *ms_out, int64_t *count_out, double *span_ms_out, int n,
                         int reset);

/*
 * Tuning and testing support.  The lattice passes split an utterance's rows
 * u into K bands, one CTA each.  The bands exchange their boundary rows
 * either inside a thread-block cluster (K <= 16; distributed shared memory)
 * or through global memory (any K; each band polls its neighbour's boundary
 * row in L2).  bands > 0 forces K for later calls: up to 16 in a cluster
 * (fewer when such a cluster does not fit the GPU) unless global exchange is
 * forced, above 16 through global memory; 0 restores the per-problem choice.
 * The results do not depend on K or on the exchange, bit for bit.
 * Process-wide; returns the previous setting.
 */
int tdt_loss_set_lattice_bands(int bands);

/*
 * Tuning and testing support: how lattice bands exchange boundary rows for
 * later calls.  mode 0: chosen per problem (global memory for lattices too
 * tall for one CTA; a cluster for forced counts up to 16), 1: always a
 * cluster (at most 16 bands), 2: always global memory.  Other values act as
 * 0.  Process-wide; returns the previous setting.
 */
int tdt_loss_set_lattice_exchange(int mode);

/*
 * Testing support for the bounded waits of the multi-band lattice passes
 * (failure detection; the pages have no counterpart).  When an utterance's
 * rows are split into K >= 2 bands, each band waits for its neighbour's
 * boundary row on every anti-diagonal, and every such wait gives up after a
 * limit: the utterance then gets a NaN loss and zero gradient rows, and the
 * call still returns normally.  With utterance >= 0, later calls run the
 * lattice passes of that utterance index with band 1 never publishing its
 * boundary row, so its neighbours' waits run out; every other utterance is
 * computed as usual.  wait_limit_cycles > 0 sets the limit of every wait of
 * later calls in GPU clock cycles (0: the default, about one second).
 * utterance < 0 switches the fault off.  Process-wide; returns the previous
 * utterance setting (-1: none).  Only multi-band lattices wait at all
 * (tdt_loss_set_lattice_bands(K >= 2), or lattices too tall for one CTA),
 * with either exchange.
 */
long long tdt_loss_test_set_halo_fault(long long utterance, long long wait_limit_cycles);

/* Human-readable text for a status code (static storage). */
const char *tdt_status_string(int status);

/* TDT_LOSS_VERSION of the loaded library. */
int tdt_loss_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TDT_LOSS_H */
