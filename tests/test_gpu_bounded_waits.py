"""The lattice's bounded waits run out, on the GPU, without a fault.

With more than one band per utterance, each band of the alpha and beta
passes waits on every anti-diagonal for its neighbour's boundary row, with a
limit on every wait.  The testing hook tdt_loss_test_set_halo_fault makes
band 1 of one chosen utterance withhold that row, so its neighbours' waits
run out after a short limit.  The call must return normally; that utterance
gets a NaN loss and zero gradient rows; every other utterance still matches
the oracle; and the next call without the fault matches the oracle again.
"""
import numpy as np
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu

LIMIT_CYCLES = 2_000_000   # about a millisecond at the GB300 clock


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _run(binding, inp, compute_grad=True):
    loss, grad = binding.tdt_loss_fwd_bwd(
        inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
        inp["blank"], inp["sigma"], "none", compute_grad=compute_grad)
    torch.cuda.synchronize()
    return loss.double().cpu().numpy(), grad


@pytest.mark.parametrize("exchange", [1, 2])
@pytest.mark.parametrize("faulted", [0, 2])
def test_wait_runs_out_and_marks_only_that_utterance(binding, oracle_mod, faulted, exchange):
    """exchange 1: bands in a thread-block cluster (mbarrier waits);
    exchange 2: bands exchanging through global memory (polled entries)."""
    w = scaled(WORKLOADS["tiny"], name="halo_fault", B=3, T=40, U=100, V=50, blank=49,
               durations=(0, 1, 2, 3), dtype="f32", std=1.0, sigma=0.05, reduction="none",
               seed=2718)
    inp = make_inputs(w, device="cuda")
    ref = oracle_mod.tdt_loss(inp["logits"].cpu().numpy(), inp["labels"].cpu().numpy(),
                              inp["logit_lens"].cpu().numpy(), inp["label_lens"].cpu().numpy(),
                              inp["durations"], inp["blank"], inp["sigma"], "none")
    prev_bands = binding.tdt_loss_set_lattice_bands(4)
    prev_mode = binding.tdt_loss_set_lattice_exchange(exchange)
    try:
        assert binding.tdt_loss_test_set_halo_fault(faulted, LIMIT_CYCLES) == -1
        try:
            loss, grad = _run(binding, inp)
            loss_only, _ = _run(binding, inp, compute_grad=False)
        finally:
            assert binding.tdt_loss_test_set_halo_fault(-1, 0) == faulted
        for b in range(w.B):
            if b == faulted:
                assert np.isnan(loss[b]) and np.isnan(loss_only[b])
                assert (grad[b] == 0).all()
            else:
                assert abs(loss[b] - ref.loss[b]) <= 1e-6 * abs(ref.loss[b])
                assert loss_only[b] == loss[b]
                err = (grad[b].double().cpu().numpy() - ref.grad[b]).__abs__().max()
                assert err <= 1e-5, err
        # the same process and GPU, fault off and default limit: every utterance matches
        loss2, grad2 = _run(binding, inp)
        assert np.all(np.abs(loss2 - ref.loss) <= 1e-6 * np.abs(ref.loss))
        assert np.abs(grad2.double().cpu().numpy() - ref.grad).max() <= 1e-5
    finally:
        binding.tdt_loss_set_lattice_bands(prev_bands)
        binding.tdt_loss_set_lattice_exchange(prev_mode)
