"""tdt_loss_fwd_bwd_noalloc: loss and gradient without any device allocation.

Some callers cannot allocate device memory while they run: a runtime that
reserved all memory at start-up and treats a later allocation as an error,
or code running while another component owns the allocator.  This entry
point takes its scratch from a fixed array inside the library instead.
Here it is called through the C ABI on two problems in a row, with and
without the gradient and with reductions mean_volume, mean_batch and none,
and each result is compared with the default entry point's and with the
float64 oracle within the parity tolerances (fp32: loss relative 1e-6,
gradient absolute 1e-5; bf16: 2e-3 / 2e-2).  A problem that needs more
scratch than the array is refused before anything is enqueued, and a child
process checks that the entry point keeps working after cudaDeviceReset (a
new context, where the array has a new address).
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-6, 1e-5), "bf16": (2e-3, 2e-2)}
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _problems(reduction=None):
    a = scaled(WORKLOADS["parakeet"], name="noalloc_f32", B=3, T=37, U=11, V=1000, blank=999,
               sigma=0.05, T_range=(20, 37), U_range=(3, 11), base_vd=1013, seed=4242)
    b = scaled(WORKLOADS["parakeet_bf16_ragged"], name="noalloc_bf16", B=4, T=60, U=17,
               V=2049, blank=2048, base_vd=2060, T_range=(30, 60), U_range=(5, 17), seed=4343)
    if reduction:
        a, b = scaled(a, reduction=reduction), scaled(b, reduction=reduction)
    return [a, b]


def _args(inp):
    return (inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"],
            inp["durations"], inp["blank"], inp["sigma"], inp["reduction"])


def _close(loss, grad, ref_loss, ref_grad, dtype):
    rtol, atol = TOL[dtype]
    l = loss.double().cpu().numpy()
    assert np.all(np.abs(l - ref_loss) <= rtol * np.abs(ref_loss)), (l, ref_loss)
    if ref_grad is not None:
        g = grad.double().cpu().numpy()
        err = np.abs(g - ref_grad).max()
        assert err <= atol, err


@pytest.mark.parametrize("compute_grad", [True, False], ids=["loss_and_grad", "loss_only"])
@pytest.mark.parametrize("reduction", [None, "none"], ids=["workload_reduction", "none"])
def test_noalloc_matches_oracle_and_default_entry_point_on_two_calls(binding, oracle_mod,
                                                                     compute_grad, reduction):
    for w in _problems(reduction):
        inp = make_inputs(w, device="cuda")
        ref_loss, ref_grad = binding.tdt_loss_fwd_bwd(*_args(inp), compute_grad=compute_grad)
        loss = torch.empty_like(ref_loss)
        grad = torch.empty_like(ref_grad) if compute_grad else None
        binding.tdt_loss_fwd_bwd_noalloc(*_args(inp), loss_out=loss, grad_out=grad,
                                         compute_grad=compute_grad)
        torch.cuda.synchronize()
        orc = oracle_mod.tdt_loss(
            inp["logits"].float().cpu().numpy(), inp["labels"].cpu().numpy(),
            inp["logit_lens"].cpu().numpy(), inp["label_lens"].cpu().numpy(), inp["durations"],
            inp["blank"], inp["sigma"], inp["reduction"], want_grad=compute_grad)
        _close(loss, grad, orc.loss, orc.grad, w.dtype)
        _close(loss, grad, ref_loss.double().cpu().numpy(),
               ref_grad.double().cpu().numpy() if compute_grad else None, w.dtype)


def test_noalloc_refuses_problems_larger_than_its_array(binding):
    so = binding.lib
    sizes = (ctypes.c_int64 * 4)(16, 750, 121, 1030)       # the large_batch shapes
    strides = (ctypes.c_int64 * 4)(750 * 121 * 1030, 121 * 1030, 1030, 1)
    durs = (ctypes.c_int32 * 5)(0, 1, 2, 3, 4)
    assert binding.tdt_loss_workspace_size([16, 750, 121, 1030], 5) > \
        binding.NOALLOC_MAX_WORKSPACE_BYTES
    f = ctypes.c_void_p(0x10000)   # never dereferenced: the call is refused first
    rc = so.tdt_loss_fwd_bwd_noalloc(f, sizes, strides, 2, f, f, f, durs, 5, 1024, 0.0, 1, f, f,
                                     None)
    assert rc == -12
    assert "fixed array" in binding.tdt_status_string(rc)


def test_noalloc_after_device_reset_in_a_child_process(binding, oracle_mod):
    """A fresh process (no PyTorch) calls the entry point, resets the device
    and calls it again in the new context; both results match the oracle."""
    r = subprocess.run([sys.executable, os.path.join(HERE, "noalloc_reset_child.py")],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().splitlines()[-1] == "OK", r.stdout + r.stderr
