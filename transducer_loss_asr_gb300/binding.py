"""ctypes binding of libtdt_loss.so (include/tdt_loss.h).

Argument marshalling only: sizes, strides, dtype codes, raw pointers and the
current CUDA stream go to the C ABI; every step of the loss runs in the
library's kernels.  PyTorch is used for device memory and streams.  There is
no fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtdt_loss.so")

DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2, "mean_batch": 3, "mean_volume": 4}

TDT_OK = 0


class TDTError(RuntimeError):
    """A TDT_ERR_* status returned by the library."""

    def __init__(self, status: int, text: str):
        super().__init__("tdt_loss status %d: %s" % (status, text))
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libtdt_loss.so is not built (%s); run `python -m transducer_loss_asr_gb300.build` "
            "or __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int
    common = [P, P, P, I, P, P, P, P, I, I, ctypes.c_double, I, P, P]
    lib.tdt_loss_fwd_bwd.restype = I
    lib.tdt_loss_fwd_bwd.argtypes = common + [P]
    lib.tdt_loss_fwd_bwd_ws.restype = I
    lib.tdt_loss_fwd_bwd_ws.argtypes = common + [P, ctypes.c_size_t, P]
    lib.tdt_loss_fwd_bwd_noalloc.restype = I
    lib.tdt_loss_fwd_bwd_noalloc.argtypes = common + [P]
    lib.tdt_rnnt_loss_fwd_bwd.restype = I
    lib.tdt_rnnt_loss_fwd_bwd.argtypes = [P, P, P, I, P, P, P, I, ctypes.c_double, I, P, P, P]
    lib.tdt_greedy_decode.restype = I
    lib.tdt_greedy_decode.argtypes = [P, P, P, I, P, P, I, I, I, P, P, P, P, P]
    lib.tdt_loss_fwd.restype = I
    lib.tdt_loss_fwd.argtypes = common[:-1] + [P, ctypes.c_size_t, P]
    lib.tdt_loss_bwd.restype = I
    lib.tdt_loss_bwd.argtypes = common[:-2] + [P, P, P, ctypes.c_size_t, P]
    lib.tdt_loss_workspace_size.restype = ctypes.c_size_t
    lib.tdt_loss_workspace_size.argtypes = [P, I]
    lib.tdt_status_string.restype = ctypes.c_char_p
    lib.tdt_status_string.argtypes = [I]
    lib.tdt_loss_version.restype = I
    lib.tdt_loss_version.argtypes = []
    lib.tdt_loss_set_lattice_bands.restype = I
    lib.tdt_loss_set_lattice_bands.argtypes = [I]
    lib.tdt_loss_set_lattice_exchange.restype = I
    lib.tdt_loss_set_lattice_exchange.argtypes = [I]
    lib.tdt_loss_test_set_halo_fault.restype = ctypes.c_longlong
    lib.tdt_loss_test_set_halo_fault.argtypes = [ctypes.c_longlong, ctypes.c_longlong]
    lib.tdt_loss_timing_enable.restype = None
    lib.tdt_loss_timing_enable.argtypes = [I]
    lib.tdt_loss_timing_read.restype = I
    lib.tdt_loss_timing_read.argtypes = [P, P, P, I, I]
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.tdt_status_string(int(status)).decode()


def _check(status: int):
    if status != TDT_OK:
        raise TDTError(status, status_string(status))


def _i64(vals):
    return (ctypes.c_int64 * 4)(*[int(v) for v in vals])


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_size(sizes, n_dur: int) -> int:
    return int(lib.tdt_loss_workspace_size(_i64(sizes), int(n_dur)))


def _marshal(logits, labels, logit_lens, label_lens, durations, blank, sigma, reduction,
             loss_out, grad_out, compute_grad, with_loss=True):
    if logits.dim() != 4:
        raise ValueError("logits must be [B, T, U+1, V+D]")
    if logits.dtype not in DTYPES:
        raise TypeError("logits dtype must be float32, float16 or bfloat16")
    B = logits.shape[0]
    dev = logits.device
    if loss_out is None and with_loss:
        loss_out = torch.empty(B if reduction == "none" else 1, dtype=torch.float32, device=dev)
    if compute_grad and grad_out is None:
        grad_out = torch.empty(logits.shape, dtype=logits.dtype, device=dev)
    if grad_out is not None and (not grad_out.is_contiguous() or grad_out.dtype != logits.dtype
                                 or tuple(grad_out.shape) != tuple(logits.shape)):
        raise ValueError("grad_out must be contiguous with the logits' shape and dtype")
    durs = (ctypes.c_int32 * len(durations))(*[int(d) for d in durations])
    args = [
        _ptr(logits), _i64(logits.shape), _i64(logits.stride()), DTYPES[logits.dtype],
        _ptr(labels) if labels is not None and labels.numel() > 0 else None,
        _ptr(logit_lens), _ptr(label_lens), durs, len(durations), int(blank), float(sigma),
        REDUCTIONS[reduction], _ptr(loss_out), _ptr(grad_out),
    ]
    for name, t in (("labels", labels), ("logit_lens", logit_lens), ("label_lens", label_lens)):
        if t is not None and (t.dtype != torch.int64 or not t.is_contiguous() or t.device != dev):
            raise ValueError("%s must be a contiguous int64 tensor on %s" % (name, dev))
    return args, loss_out, grad_out


def tdt_loss_fwd_bwd(logits, labels, logit_lens, label_lens, durations, blank, sigma=0.0,
                     reduction="mean_volume", loss_out=None, grad_out=None, compute_grad=True):
    """TDT loss and its gradient in one call on the current CUDA stream.

    Returns (loss, grad): loss float32 [B] ("none") or [1]; grad with the
    logits' shape and dtype (None when compute_grad is False and no grad_out
    is given).  ``logits`` may be a strided view such as ``base[..., :V+D]``.
    """
    args, loss_out, grad_out = _marshal(logits, labels, logit_lens, label_lens, durations,
                                        blank, sigma, reduction, loss_out, grad_out,
                                        compute_grad)
    with torch.cuda.device(logits.device):
        _check(lib.tdt_loss_fwd_bwd(*args, _stream_handle(logits.device)))
    return loss_out, grad_out


def tdt_rnnt_loss_fwd_bwd(logits, labels, logit_lens, label_lens, blank, sigma=0.0,
                          reduction="mean_volume", loss_out=None, grad_out=None,
                          compute_grad=True):
    """Plain RNN-T loss (no duration head) and its gradient on the current
    CUDA stream: logits [B, T, U+1, V]; other arguments as tdt_loss_fwd_bwd
    without durations.  Returns (loss, grad)."""
    args, loss_out, grad_out = _marshal(logits, labels, logit_lens, label_lens, [0], blank,
                                        sigma, reduction, loss_out, grad_out, compute_grad)
    # drop the durations pointer and count of the TDT argument list
    rargs = args[:7] + args[9:]
    with torch.cuda.device(logits.device):
        _check(lib.tdt_rnnt_loss_fwd_bwd(*rargs, _stream_handle(logits.device)))
    return loss_out, grad_out


def tdt_greedy_decode(logits, logit_lens, durations, blank, max_symbols=10):
    """Greedy TDT decoding of joint outputs ``logits`` [B, T, U+1, V+D] on the
    current CUDA stream.  Returns (n [B], tokens, frames, token_durations
    [B, U+1]) as int32 CUDA tensors, -1 past n[b]."""
    if logits.dim() != 4:
        raise ValueError("logits must be [B, T, U+1, V+D]")
    if logits.dtype not in DTYPES:
        raise TypeError("logits dtype must be float32, float16 or bfloat16")
    if logit_lens.dtype != torch.int64 or logit_lens.device != logits.device:
        raise ValueError("logit_lens must be an int64 tensor on %s" % logits.device)
    B, _, U1, _ = logits.shape
    dev = logits.device
    n = torch.empty(B, dtype=torch.int32, device=dev)
    tok, frm, dur = (torch.empty(B, U1, dtype=torch.int32, device=dev) for _ in range(3))
    durs = (ctypes.c_int32 * len(durations))(*[int(d) for d in durations])
    with torch.cuda.device(dev):
        _check(lib.tdt_greedy_decode(
            _ptr(logits), _i64(logits.shape), _i64(logits.stride()), DTYPES[logits.dtype],
            _ptr(logit_lens.contiguous()), durs, len(durations), int(blank), int(max_symbols),
            _ptr(n), _ptr(tok), _ptr(frm), _ptr(dur), _stream_handle(dev)))
    return n, tok, frm, dur


def tdt_loss_fwd_bwd_ws(logits, labels, logit_lens, label_lens, durations, blank, workspace,
                        sigma=0.0, reduction="mean_volume", loss_out=None, grad_out=None,
                        compute_grad=True):
    """As tdt_loss_fwd_bwd with a caller-owned uint8 CUDA workspace tensor."""
    args, loss_out, grad_out = _marshal(logits, labels, logit_lens, label_lens, durations,
                                        blank, sigma, reduction, loss_out, grad_out,
                                        compute_grad)
    with torch.cuda.device(logits.device):
        _check(lib.tdt_loss_fwd_bwd_ws(*args, _ptr(workspace), workspace.numel(),
                                       _stream_handle(logits.device)))
    return loss_out, grad_out


NOALLOC_MAX_WORKSPACE_BYTES = 64 * 1024 * 1024


def tdt_loss_fwd_bwd_noalloc(logits, labels, logit_lens, label_lens, durations, blank,
                             sigma=0.0, reduction="mean_volume", loss_out=None, grad_out=None,
                             compute_grad=True):
    """As tdt_loss_fwd_bwd, for callers that cannot allocate device memory.

    The library allocates nothing: its scratch is a fixed 64 MiB device array
    inside the library (problems needing more are rejected); every call on a
    device shares it, so order the calls on one stream.  Only the outputs
    are created here when not given -- pass loss_out and grad_out to
    allocate nothing at all.
    """
    args, loss_out, grad_out = _marshal(logits, labels, logit_lens, label_lens, durations,
                                        blank, sigma, reduction, loss_out, grad_out,
                                        compute_grad)
    with torch.cuda.device(logits.device):
        _check(lib.tdt_loss_fwd_bwd_noalloc(*args, _stream_handle(logits.device)))
    return loss_out, grad_out


def _new_workspace(logits, n_dur):
    return torch.empty(max(1, workspace_size(logits.shape, n_dur)), dtype=torch.uint8,
                       device=logits.device)


def tdt_loss_fwd(logits, labels, logit_lens, label_lens, durations, blank, sigma=0.0,
                 reduction="mean_volume", loss_out=None, workspace=None):
    """Forward half of the split API: returns (loss, workspace).

    The workspace (a uint8 CUDA tensor, created when not given) holds what
    tdt_loss_bwd needs; keep it untouched until then.
    """
    args, loss_out, _ = _marshal(logits, labels, logit_lens, label_lens, durations, blank, sigma,
                                 reduction, loss_out, None, False)
    if workspace is None:
        workspace = _new_workspace(logits, len(durations))
    with torch.cuda.device(logits.device):
        _check(lib.tdt_loss_fwd(*args[:-1], _ptr(workspace), workspace.numel(),
                                _stream_handle(logits.device)))
    return loss_out, workspace


def tdt_loss_bwd(logits, labels, logit_lens, label_lens, durations, blank, workspace,
                 grad_loss=None, sigma=0.0, reduction="mean_volume", grad_out=None):
    """Backward half: the gradient for upstream gradient ``grad_loss``.

    ``grad_loss``: float32 CUDA tensor with B elements ("none") or one
    element, or None for 1.  Arguments other than grad_loss/grad_out must be
    those of the tdt_loss_fwd call that filled ``workspace``.  ``grad_out``
    may be ``logits`` itself (contiguous logits): the gradient then replaces
    them.
    """
    B = logits.shape[0]
    if grad_loss is not None:
        want = B if reduction == "none" else 1
        if (grad_loss.dtype != torch.float32 or not grad_loss.is_contiguous()
                or grad_loss.numel() != want or grad_loss.device != logits.device):
            raise ValueError("grad_loss must be a contiguous float32 tensor of %d element(s) "
                             "on %s" % (want, logits.device))
    args, _, grad_out = _marshal(logits, labels, logit_lens, label_lens, durations, blank, sigma,
                                 reduction, None, grad_out, True, with_loss=False)
    with torch.cuda.device(logits.device):
        _check(lib.tdt_loss_bwd(*args[:-2], _ptr(grad_loss), args[-1], _ptr(workspace),
                                workspace.numel(), _stream_handle(logits.device)))
    return grad_out


def tdt_loss_workspace_size(sizes, n_dur: int) -> int:
    """Bytes of scratch tdt_loss_fwd_bwd_ws needs (0 for invalid sizes)."""
    return workspace_size(sizes, n_dur)


def tdt_status_string(status: int) -> str:
    return status_string(status)


def tdt_loss_version() -> int:
    return int(lib.tdt_loss_version())


def tdt_loss_set_lattice_bands(bands: int) -> int:
    """Force K bands (CTAs per utterance and direction) in the lattice passes;
    0 = automatic.  Results do not depend on K.  Returns the previous value."""
    return int(lib.tdt_loss_set_lattice_bands(int(bands)))


def tdt_loss_set_lattice_exchange(mode: int) -> int:
    """How lattice bands exchange boundary rows: 0 = automatic, 1 = a
    thread-block cluster, 2 = global memory.  Results do not depend on it.
    Returns the previous value."""
    return int(lib.tdt_loss_set_lattice_exchange(int(mode)))


def tdt_loss_test_set_halo_fault(utterance: int, wait_limit_cycles: int = 0) -> int:
    """Testing: make the multi-band lattice passes of utterance index
    ``utterance`` lose their band-1 boundary row so the neighbours' bounded
    waits run out (NaN loss, zero gradient rows for that utterance only);
    ``wait_limit_cycles`` > 0 shortens every wait's limit.  utterance < 0
    switches it off.  Returns the previous utterance setting."""
    return int(lib.tdt_loss_test_set_halo_fault(int(utterance), int(wait_limit_cycles)))


KERNEL_NAMES = ("node_tables", "lattice", "reduce", "grad")


def tdt_loss_timing_enable(on: bool) -> None:
    """Record CUDA events around each kernel of later calls (benchmarks only)."""
    lib.tdt_loss_timing_enable(1 if on else 0)


def tdt_loss_timing_read(reset: bool = True):
    """{kernel name: (summed ms, launches, summed busy-window ms)} since the
    last reset; waits for the events.  The busy window of a kernel in one call
    runs from the start of its first launch to the end of its last (launches
    on several streams may overlap)."""
    n = len(KERNEL_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    span = (ctypes.c_double * n)()
    rc = lib.tdt_loss_timing_read(ms, cnt, span, n, 1 if reset else 0)
    if rc < 0:
        raise TDTError(rc, status_string(rc))
    return {KERNEL_NAMES[i]: (ms[i], cnt[i], span[i]) for i in range(n)}
