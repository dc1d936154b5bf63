"""CPU oracle for the Token-and-Duration Transducer (TDT) loss -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``transducer_loss_asr_gb300``) never imports it, and this package imports
nothing from the product: the two share no code.

The arithmetic lives in ``tdt_oracle.c`` (the TDT loss) and
``rnnt_oracle.c`` (the plain RNN-T loss, no duration head), plain float64 C
with OpenMP only over independent utterances and nodes; this module compiles
them with gcc and marshals numpy arrays into them.  See the header of ``tdt_oracle.c`` for the
passages of "tdt-loss: add TDT loss kernel" (kernels-community PR #882) and
"Add TDT loss kernel" (transformers PR #46048) that it follows, and for the
reading of the lattice it writes out.

Every function here is pinned by the ``-m "not gpu"`` tests: brute-force
enumeration of alignment paths, a linear-system (path-sum) formulation,
closed forms for uniform logits, central finite differences and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tdt_oracle.c")
_SRCS = (_SRC, os.path.join(_HERE, "rnnt_oracle.c"))
_LIB_PATH = os.path.join(_HERE, "libtdt_oracle.so")
_lock = threading.Lock()
_lib = None

REDUCTIONS = {"none": 0, "sum": 1, "mean": 2, "mean_batch": 3, "mean_volume": 4}


def build(force: bool = False) -> str:
    """Compile tdt_oracle.c and rnnt_oracle.c into libtdt_oracle.so next to
    them (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library (the default one, or a test's variant)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.tdt_oracle_run.restype = ctypes.c_int
    lib.tdt_oracle_run.argtypes = [
        P, ctypes.c_int, P, P, P, I64, P, P, P, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_int, P, P, P, P, P, P, P, P, I64, P]
    lib.tdt_oracle_tables.restype = ctypes.c_int
    lib.tdt_oracle_tables.argtypes = [
        P, ctypes.c_int, P, P, P, I64, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P]
    if hasattr(lib, "rnnt_oracle_run"):  # absent from single-file test variants
        lib.rnnt_oracle_run.restype = ctypes.c_int
        lib.rnnt_oracle_run.argtypes = [
            P, ctypes.c_int, P, P, P, I64, P, P, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            P, P, P, P, P, P, P, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class OracleResult:
    loss: np.ndarray          # [B] for reduction "none", else [1]
    utt_loss: np.ndarray      # [B] per-utterance L_b
    scale: np.ndarray         # [B] c_b
    ll_alpha: np.ndarray      # [B] log-likelihood from the alpha pass
    ll_beta: np.ndarray       # [B] beta(0, 0)
    alpha: np.ndarray | None  # [B, T, U1]
    beta: np.ndarray | None   # [B, T, U1]
    grad: np.ndarray | None   # [B, T, U1, V+D] or [n_rows, V+D]


def _logits_view(logits: np.ndarray):
    if logits.dtype == np.float64:
        f64 = 1
    elif logits.dtype == np.float32:
        f64 = 0
    else:
        raise TypeError("oracle logits must be float32 (an exact up-cast) or float64")
    if logits.ndim != 4:
        raise ValueError("logits must be [B, T, U+1, V+D]")
    strides = np.array([s // logits.itemsize for s in logits.strides], dtype=np.int64)
    if any(s * logits.itemsize != s_b for s, s_b in zip(strides, logits.strides)):
        raise ValueError("logits strides must be whole elements")
    # Base pointer of the view (numpy's data pointer already points at [0,0,0,0]).
    return f64, strides


def tdt_loss(logits: np.ndarray, labels: np.ndarray, logit_lens: np.ndarray,
             label_lens: np.ndarray, durations, blank: int, sigma: float = 0.0,
             reduction: str = "mean_volume", want_grad: bool = True, rows=None,
             want_lattice: bool = False, lib=None) -> OracleResult:
    """Evaluate loss (and gradient) of the TDT loss in float64 on the CPU.

    logits: float32/float64 array [B, T, U+1, V+D], any element strides
    (a slice ``base[..., :V+D]`` works without a copy).  labels: int64
    [B, >= U] (entries past label_lens ignored).  rows: optional flat node
    ids ``(b*T + t)*(U+1) + u``; the gradient is then returned for those rows
    only, shape [len(rows), V+D].  lib: a library from ``load_library``
    (default: the oracle built from tdt_oracle.c).
    """
    lib = _load() if lib is None else lib
    f64, strides = _logits_view(logits)
    B, T, U1, VD = logits.shape
    sizes = np.array([B, T, U1, VD], dtype=np.int64)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    if labels.ndim != 2 or labels.shape[0] != B:
        raise ValueError("labels must be [B, U]")
    labels_stride = labels.shape[1]
    if labels_stride < U1 - 1:
        raise ValueError("labels must have at least U = sizes[2] - 1 columns")
    if labels_stride == 0:
        labels = np.zeros((B, 1), dtype=np.int64)
        labels_stride = 1
    logit_lens = np.ascontiguousarray(logit_lens, dtype=np.int64)
    label_lens = np.ascontiguousarray(label_lens, dtype=np.int64)
    dur = np.ascontiguousarray(np.asarray(durations, dtype=np.int32))
    red = REDUCTIONS[reduction]
    loss = np.zeros(B if red == 0 else 1, dtype=np.float64)
    utt = np.zeros(B, dtype=np.float64)
    scale = np.zeros(B, dtype=np.float64)
    lla = np.zeros(B, dtype=np.float64)
    llb = np.zeros(B, dtype=np.float64)
    alpha = np.zeros((B, T, U1), dtype=np.float64) if want_lattice else None
    beta = np.zeros((B, T, U1), dtype=np.float64) if want_lattice else None
    grad = None
    rows_arr = None
    n_rows = 0
    if want_grad:
        if rows is None:
            grad = np.zeros((B, T, U1, VD), dtype=np.float64)
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            n_rows = rows_arr.size
            grad = np.zeros((n_rows, VD), dtype=np.float64)
    rc = lib.tdt_oracle_run(
        logits.ctypes.data_as(ctypes.c_void_p), f64, _ptr(sizes), _ptr(strides), _ptr(labels),
        labels_stride, _ptr(logit_lens), _ptr(label_lens), _ptr(dur), int(dur.size), int(blank),
        float(sigma), red, _ptr(loss), _ptr(utt), _ptr(scale), _ptr(alpha), _ptr(beta),
        _ptr(lla), _ptr(llb), _ptr(rows_arr), n_rows, _ptr(grad))
    if rc != 0:
        raise ValueError("tdt_oracle_run rejected its arguments (status %d)" % rc)
    return OracleResult(loss, utt, scale, lla, llb, alpha, beta, grad)


def rnnt_loss(logits: np.ndarray, labels: np.ndarray, logit_lens: np.ndarray,
              label_lens: np.ndarray, blank: int, sigma: float = 0.0,
              reduction: str = "mean_volume", want_grad: bool = True,
              want_lattice: bool = False, lib=None) -> OracleResult:
    """Plain RNN-T loss (no duration head) and its gradient in float64
    (rnnt_oracle.c).  logits [B, T, U+1, V], any element strides; the other
    arguments as for tdt_loss.  grad has the logits' shape."""
    lib = _load() if lib is None else lib
    f64, strides = _logits_view(logits)
    B, T, U1, V = logits.shape
    sizes = np.array([B, T, U1, V], dtype=np.int64)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    if labels.ndim != 2 or labels.shape[0] != B or labels.shape[1] < U1 - 1:
        raise ValueError("labels must be [B, >= U]")
    lstride = labels.shape[1]
    if lstride == 0:
        labels = np.zeros((B, 1), dtype=np.int64)
        lstride = 1
    logit_lens = np.ascontiguousarray(logit_lens, dtype=np.int64)
    label_lens = np.ascontiguousarray(label_lens, dtype=np.int64)
    red = REDUCTIONS[reduction]
    loss = np.zeros(B if red == 0 else 1)
    utt = np.zeros(B); scale = np.zeros(B); lla = np.zeros(B); llb = np.zeros(B)
    alpha = np.zeros((B, T, U1)) if want_lattice else None
    beta = np.zeros((B, T, U1)) if want_lattice else None
    grad = np.zeros((B, T, U1, V)) if want_grad else None
    rc = lib.rnnt_oracle_run(
        logits.ctypes.data_as(ctypes.c_void_p), f64, _ptr(sizes), _ptr(strides), _ptr(labels),
        lstride, _ptr(logit_lens), _ptr(label_lens), int(blank), float(sigma), red,
        _ptr(loss), _ptr(utt), _ptr(scale), _ptr(alpha), _ptr(beta), _ptr(lla), _ptr(llb),
        _ptr(grad))
    if rc != 0:
        raise ValueError("rnnt_oracle_run rejected its arguments (status %d)" % rc)
    return OracleResult(loss, utt, scale, lla, llb, alpha, beta, grad)


def node_tables(logits: np.ndarray, labels: np.ndarray, logit_lens: np.ndarray,
                label_lens: np.ndarray, n_dur: int, blank: int):
    """Per-node log-softmax tables: (lse_tok, lp_blank, lp_label, lp_dur[..., D])."""
    lib = _load()
    f64, strides = _logits_view(logits)
    B, T, U1, VD = logits.shape
    sizes = np.array([B, T, U1, VD], dtype=np.int64)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    if labels.shape[1] == 0:
        labels = np.zeros((B, 1), dtype=np.int64)
    logit_lens = np.ascontiguousarray(logit_lens, dtype=np.int64)
    label_lens = np.ascontiguousarray(label_lens, dtype=np.int64)
    lse = np.zeros((B, T, U1)); lpb = np.zeros((B, T, U1)); lpl = np.zeros((B, T, U1))
    lpd = np.zeros((B, T, U1, n_dur))
    rc = lib.tdt_oracle_tables(
        logits.ctypes.data_as(ctypes.c_void_p), f64, _ptr(sizes), _ptr(strides), _ptr(labels),
        labels.shape[1], _ptr(logit_lens), _ptr(label_lens), int(n_dur), int(blank), _ptr(lse),
        _ptr(lpb), _ptr(lpl), _ptr(lpd))
    if rc != 0:
        raise ValueError("tdt_oracle_tables rejected its arguments (status %d)" % rc)
    return lse, lpb, lpl, lpd
