"""Child process of tests/test_zz_no_alloc.py: the allocation-free entry point
across cudaDeviceReset, with no PyTorch in the process.

It calls tdt_loss_fwd_bwd_noalloc, resets the device, and calls it again in
the new context, checking both results against the float64 oracle.  Before
the second call it checks, through the driver, that the current context's
unique id changed: that id is what makes the library look up its scratch
array again, so the second call only runs when that precondition holds
(otherwise the child prints SKIP).  Prints OK on success.
"""
import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

LIB = os.path.join(ROOT, "transducer_loss_asr_gb300", "libtdt_loss.so")


def main():
    lib = ctypes.CDLL(LIB)  # loads the CUDA runtime it was linked with
    try:
        rt = ctypes.CDLL("libcudart.so.13")
    except OSError:
        rt = ctypes.CDLL("/usr/local/cuda/lib64/libcudart.so.13")
    drv = ctypes.CDLL("libcuda.so.1")
    P = ctypes.c_void_p

    def ok(rc, what):
        if rc != 0:
            raise RuntimeError("%s failed: %d" % (what, rc))

    def ctx_id():
        ctx = P()
        ok(drv.cuCtxGetCurrent(ctypes.byref(ctx)), "cuCtxGetCurrent")
        if not ctx.value:
            return None
        cid = ctypes.c_ulonglong()
        ok(drv.cuCtxGetId(ctx, ctypes.byref(cid)), "cuCtxGetId")
        return cid.value

    rng = np.random.default_rng(99)
    B, T, U, V, durs = 2, 20, 6, 50, [0, 1, 2]
    D = len(durs)
    z = rng.standard_normal((B, T, U + 1, V + D)).astype(np.float32)
    labels = rng.integers(0, V - 1, (B, U)).astype(np.int64)
    tl = np.array([T, 15], dtype=np.int64)
    ul = np.array([U, 4], dtype=np.int64)
    labels[1, 4:] = -100
    blank, sigma, red = V - 1, 0.05, 0  # reduction none
    ref = oracle.tdt_loss(z, labels, tl, ul, durs, blank, sigma, "none")

    lib.tdt_loss_fwd_bwd_noalloc.restype = ctypes.c_int
    lib.tdt_loss_fwd_bwd_noalloc.argtypes = [
        P, P, P, ctypes.c_int, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        ctypes.c_int, P, P, P]
    sizes = (ctypes.c_int64 * 4)(B, T, U + 1, V + D)
    strides = (ctypes.c_int64 * 4)(T * (U + 1) * (V + D), (U + 1) * (V + D), V + D, 1)
    cdurs = (ctypes.c_int32 * D)(*durs)

    def one_call():
        host = [z, labels, tl, ul]
        dev = []
        for a in host:
            p = P()
            ok(rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(a.nbytes)), "cudaMalloc")
            ok(rt.cudaMemcpy(p, a.ctypes.data_as(P), ctypes.c_size_t(a.nbytes), 1), "H2D")
            dev.append(p)
        loss_d, grad_d = P(), P()
        ok(rt.cudaMalloc(ctypes.byref(loss_d), ctypes.c_size_t(4 * B)), "cudaMalloc")
        ok(rt.cudaMalloc(ctypes.byref(grad_d), ctypes.c_size_t(z.nbytes)), "cudaMalloc")
        rc = lib.tdt_loss_fwd_bwd_noalloc(dev[0], sizes, strides, 0, dev[1], dev[2], dev[3],
                                          cdurs, D, blank, sigma, red, loss_d, grad_d, None)
        ok(rc, "tdt_loss_fwd_bwd_noalloc")
        ok(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
        loss = np.zeros(B, dtype=np.float32)
        grad = np.zeros_like(z)
        ok(rt.cudaMemcpy(loss.ctypes.data_as(P), loss_d, ctypes.c_size_t(4 * B), 2), "D2H")
        ok(rt.cudaMemcpy(grad.ctypes.data_as(P), grad_d, ctypes.c_size_t(z.nbytes), 2), "D2H")
        for p in dev + [loss_d, grad_d]:
            ok(rt.cudaFree(p), "cudaFree")
        rel = np.abs(loss.astype(np.float64) - ref.loss) / np.abs(ref.loss)
        err = np.abs(grad.astype(np.float64) - ref.grad).max()
        if not (rel.max() <= 1e-6 and err <= 1e-5):
            raise AssertionError("mismatch: loss rel %.3e grad %.3e" % (rel.max(), err))

    ok(rt.cudaSetDevice(0), "cudaSetDevice")
    ok(rt.cudaFree(None), "cudaFree(0)")  # the child (not the library) creates the context
    before = ctx_id()
    one_call()
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    ok(rt.cudaSetDevice(0), "cudaSetDevice")
    ok(rt.cudaFree(None), "cudaFree(0)")
    after = ctx_id()
    if before is None or after is None or before == after:
        print("SKIP context id unchanged across the reset: %s %s" % (before, after))
        return 0
    one_call()
    print("OK")
    return 0


if __name__ == "__main__":
    sys.exit(main())
