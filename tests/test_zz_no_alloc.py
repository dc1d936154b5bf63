"""tdt_loss_fwd_bwd_noalloc: loss and gradient without any device allocation.

Some callers cannot allocate device memory while they run (a runtime that
reserved all memory at start-up, or code running while another component
owns the allocator).  This entry point takes its scratch from a fixed array
inside the library instead.  Here it is called through the C ABI twice in a
row, on two different problems, and each result is compared with the
default entry point's within the parity tolerances (fp32: loss relative
1e-6, gradient absolute 1e-5; bf16: 2e-3 / 2e-2).  A problem that needs more
scratch than the array is refused before anything is enqueued.
"""
import ctypes

import numpy as np
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-6, 1e-5), "bf16": (2e-3, 2e-2)}


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _problems():
    a = scaled(WORKLOADS["parakeet"], name="noalloc_f32", B=3, T=37, U=11, V=1000, blank=999,
               sigma=0.05, T_range=(20, 37), U_range=(3, 11), base_vd=1013, seed=4242)
    b = scaled(WORKLOADS["parakeet_bf16_ragged"], name="noalloc_bf16", B=4, T=60, U=17,
               V=2049, blank=2048, base_vd=2060, T_range=(30, 60), U_range=(5, 17), seed=4343)
    return [a, b]


def _args(inp):
    return (inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"],
            inp["durations"], inp["blank"], inp["sigma"], inp["reduction"])


def test_noalloc_matches_default_entry_point_on_two_calls(binding):
    for w in _problems():
        inp = make_inputs(w, device="cuda")
        ref_loss, ref_grad = binding.tdt_loss_fwd_bwd(*_args(inp))
        loss = torch.empty_like(ref_loss)
        grad = torch.empty_like(ref_grad)
        binding.tdt_loss_fwd_bwd_noalloc(*_args(inp), loss_out=loss, grad_out=grad)
        torch.cuda.synchronize()
        rtol, atol = TOL[w.dtype]
        l, lr = loss.double().cpu().numpy(), ref_loss.double().cpu().numpy()
        assert np.all(np.abs(l - lr) <= rtol * np.abs(lr)), (l, lr)
        err = (grad.double() - ref_grad.double()).abs().max().item()
        assert err <= atol, err


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
