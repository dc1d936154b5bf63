"""Per-kernel timing of the fused call (benchmark support), on the GPU.

Problems whose logits reach 8 MiB run the chunked schedule: one K1
node-table pass, one lattice pass and one K4 gradient pass per chunk (up to
four chunks of utterances) and one reduction.  Smaller ones run each kernel
once, serially on the caller's stream.  The timing read returns, per kernel,
the summed launch durations, the number of launches and the summed per-call
busy window (first launch start to last launch end).  Checked: launch
counts on both paths, positive times, a busy window at least as long as an
average launch, and the reset.
"""
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


@pytest.mark.parametrize("V,per_launch", [(8193, 4), (513, 1)], ids=["chunked", "serial"])
def test_timing_counts_and_busy_windows(binding, V, per_launch):
    w = scaled(WORKLOADS["parakeet"], name="timing", B=4, T=40, U=8, V=V, blank=V - 1)
    inp = make_inputs(w, device="cuda")
    calls = 3
    binding.tdt_loss_timing_read(reset=True)
    binding.tdt_loss_timing_enable(True)
    try:
        for _ in range(calls):
            binding.tdt_loss_fwd_bwd(inp["logits"], inp["labels"], inp["logit_lens"],
                                     inp["label_lens"], inp["durations"], inp["blank"],
                                     inp["sigma"], inp["reduction"])
        torch.cuda.synchronize()
        kt = binding.tdt_loss_timing_read(reset=True)
    finally:
        binding.tdt_loss_timing_enable(False)
    per_call = {"node_tables": per_launch, "lattice": per_launch, "reduce": 1,
                "grad": per_launch}
    for name, n in per_call.items():
        ms, launches, busy = kt[name]
        assert launches == n * calls, (name, launches)
        assert ms > 0.0 and busy > 0.0, name
        assert busy >= ms / launches * 0.999, (name, ms, launches, busy)
    again = binding.tdt_loss_timing_read(reset=True)
    assert all(v == (0.0, 0, 0.0) for v in again.values())
