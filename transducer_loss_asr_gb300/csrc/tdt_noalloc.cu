// tdt_noalloc.cu -- tdt_loss_fwd_bwd_noalloc: the loss and gradient with no
// device allocation at all, for callers that cannot allocate.
//
// Some callers of a loss cannot call cudaMalloc or any allocator: code that
// runs while another component owns the device memory pool and forbids
// allocation, runtimes that preallocate everything at start-up and treat a
// later allocation as an error, or embedders that must not grow the
// process's device footprint during training.  For them the scratch lives in
// a fixed file-scope device array, allocated when the CUDA module holding it
// is loaded and held until the process exits.  The caller still passes the
// inputs and the outputs.
//
// Differences from tdt_loss_fwd_bwd:
//  - the scratch is kNoAllocScratchBytes (64 MiB) at most; a call whose
//    tdt_loss_workspace_size exceeds that is rejected with
//    TDT_ERR_NOALLOC_TOO_LARGE before anything is enqueued;
//  - the kernels run one after another on the caller's stream (no internal
//    stream and no events are created);
//  - every call on a device shares the same array: two calls whose work
//    overlaps on the GPU (different streams, or different host threads
//    without ordering) race on it.  Order them on one stream.  No entry of
//    the array needs to start at zero: every entry a call reads is written
//    earlier in the same call, so what the previous call left there is
//    never used.
//  - the first call in each CUDA context (the first call on a device, and
//    the first one after cudaDeviceReset or in another context) looks up
//    the array's device address (cudaGetSymbolAddress, with that context
//    current) and caches it under the context's unique id; make that first
//    call before any stream capture.
#include <cuda.h>

#include <mutex>

#include "../../include/tdt_loss.h"
#include "tdt_common.cuh"

namespace tdt {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)TDT_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The address is valid only in the context it was looked up in: a device
// reset (or another context made current on the same device) loads the
// module again, possibly elsewhere.  So each device's entry remembers the
// unique id of its context (cuCtxGetId, reached through the runtime's
// driver entry point, so no link to the driver library is needed).
struct ScratchEntry {
  unsigned long long ctx_id = 0;  // 0: no lookup yet
  void *addr = nullptr;
};

std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the context current on this thread; 0 when none is current
// or the driver cannot tell.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context: cached per
// device under the context's id, looked up again (with that context
// current) whenever the id differs.  nullptr on failure.
void *scratch_in_current_context() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> g(g_mu);
  unsigned long long id = current_context_id();
  ScratchEntry &e = g_scratch[dev];
  if (id != 0 && e.ctx_id == id && e.addr) return e.addr;
  void *ptr = nullptr;
  // also makes the device's primary context current if none was
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
  if (id == 0) id = current_context_id();
  if (id == 0) return ptr;  // no id to key on: use the fresh address, cache nothing
  e.ctx_id = id;
  e.addr = ptr;
  return ptr;
}

}  // namespace
}  // namespace tdt

extern "C" int tdt_loss_fwd_bwd_noalloc(const void *logits, const int64_t sizes[4],
                                        const int64_t strides[4], int dtype,
                                        const int64_t *labels, const int64_t *logit_lens,
                                        const int64_t *label_lens, const int32_t *durations,
                                        int n_dur, int blank, double sigma, int reduction,
                                        float *loss_out, void *grad_out, void *stream) {
  tdt::Problem p;
  int rc = tdt::validate(logits, sizes, strides, dtype, labels, logit_lens, label_lens,
                         durations, n_dur, blank, sigma, reduction, loss_out, grad_out, &p, true);
  if (rc != TDT_OK) return rc;
  p.gx_rows = tdt::lattice_global_rows(p, p.B);
  tdt::Layout L;
  if (!tdt::make_layout(sizes, n_dur, &L)) return TDT_ERR_BAD_SIZES;
  if (L.total > tdt::kNoAllocScratchBytes) return TDT_ERR_NOALLOC_TOO_LARGE;
  void *scratch = tdt::scratch_in_current_context();
  if (!scratch) return TDT_ERR_CUDA;
  const tdt::Workspace ws = tdt::carve(L, scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long rows = p.B * p.T * p.U1;
  const bool with_grad = grad_out != nullptr;
  if (tdt::launch_node_tables(p, dtype, ws, 0, rows, s) != cudaSuccess) return TDT_ERR_CUDA;
  if (tdt::launch_lattice(p, ws, 0, p.B, with_grad, s) != cudaSuccess) return TDT_ERR_CUDA;
  if (tdt::launch_reduce(p, ws, loss_out, s) != cudaSuccess) return TDT_ERR_CUDA;
  if (with_grad && tdt::launch_grad(p, dtype, ws, grad_out, nullptr, 0, rows, s) != cudaSuccess)
    return TDT_ERR_CUDA;
  return TDT_OK;
}
