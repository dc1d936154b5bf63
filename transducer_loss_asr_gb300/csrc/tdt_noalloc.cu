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
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture.
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

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current).  nullptr on failure.
void *scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
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
  tdt::Layout L;
  if (!tdt::make_layout(sizes, n_dur, &L)) return TDT_ERR_BAD_SIZES;
  if (L.total > tdt::kNoAllocScratchBytes) return TDT_ERR_NOALLOC_TOO_LARGE;
  void *scratch = tdt::scratch_on_current_device();
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
