"""Plain RNN-T loss (no duration head) on the GPU (tdt_rnnt_loss_fwd_bwd)
against the float64 RNN-T oracle, element by element.  Same tolerances as
the TDT parity tests: fp32 loss relative <= 1e-6, gradient absolute <= 1e-5;
bf16/fp16 loss relative <= 2e-3, gradient absolute <= 2e-2."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-6, 1e-5), torch.bfloat16: (2e-3, 2e-2), torch.float16: (2e-3, 2e-2)}


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _make(seed, B, T, U, V, blank, dtype, std=1.0, ragged=True, base_v=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    W = base_v or V
    z = (torch.randn(B, T, U + 1, W, generator=g, device="cuda") * std).to(dtype)
    if base_v:
        z = z[..., :V]
    c = np.random.default_rng(seed)
    tl = c.integers(max(1, T // 2), T + 1, size=B) if ragged else np.full(B, T)
    ul = c.integers(0, U + 1, size=B) if ragged else np.full(B, U)
    labels = np.full((B, U), -100, dtype=np.int64)
    for b in range(B):
        y = c.integers(0, V - 1, size=ul[b])
        labels[b, : ul[b]] = y + (y >= blank)
    return (z, torch.from_numpy(labels).cuda(), torch.from_numpy(tl).cuda(),
            torch.from_numpy(ul).cuda())


def _check(binding, oracle_mod, z, labels, tl, ul, blank, sigma, reduction, grad_out=None):
    loss, grad = binding.tdt_rnnt_loss_fwd_bwd(z, labels, tl, ul, blank, sigma, reduction,
                                               grad_out=grad_out)
    torch.cuda.synchronize()
    ref = oracle_mod.rnnt_loss(z.float().cpu().numpy(), labels.cpu().numpy(), tl.cpu().numpy(),
                               ul.cpu().numpy(), blank, sigma, reduction)
    rtol, atol = TOL[z.dtype]
    l = loss.double().cpu().numpy()
    fin = np.isfinite(ref.loss)
    assert np.array_equal(np.isnan(l), np.isnan(ref.loss))
    rel = np.abs(l[fin] - ref.loss[fin]) / np.maximum(np.abs(ref.loss[fin]), 1e-30)
    assert rel.size == 0 or rel.max() <= rtol, rel.max()
    err = np.abs(grad.double().cpu().numpy() - ref.grad)
    assert err.max() <= atol, err.max()
    return loss, grad


CASES = {
    "f32_small": dict(B=3, T=17, U=6, V=40, blank=39, dtype=torch.float32, sigma=0.0),
    "f32_ragged_view": dict(B=4, T=33, U=12, V=1000, blank=0, dtype=torch.float32, sigma=0.05,
                            base_v=1011),
    "bf16_ragged": dict(B=4, T=40, U=20, V=513, blank=512, dtype=torch.bfloat16, sigma=0.0,
                        std=1.5),
    "f16_full": dict(B=2, T=25, U=9, V=129, blank=128, dtype=torch.float16, sigma=0.1,
                     ragged=False),
    "f32_long_rows": dict(B=1, T=6, U=3, V=20001, blank=20000, dtype=torch.float32, sigma=0.0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_rnnt_parity(binding, oracle_mod, name):
    c = dict(CASES[name])
    sigma, dtype = c.pop("sigma"), c.pop("dtype")
    std, ragged, base_v = c.pop("std", 1.0), c.pop("ragged", True), c.pop("base_v", None)
    z, labels, tl, ul = _make(101, c["B"], c["T"], c["U"], c["V"], c["blank"], dtype, std,
                              ragged, base_v)
    _check(binding, oracle_mod, z, labels, tl, ul, c["blank"], sigma, "mean_volume")


@pytest.mark.parametrize("red", ["none", "sum", "mean", "mean_batch", "mean_volume"])
def test_rnnt_reductions(binding, oracle_mod, red):
    z, labels, tl, ul = _make(7, 5, 15, 6, 33, 32, torch.float32)
    ul = torch.clamp(ul, min=1)
    _check(binding, oracle_mod, z, labels, tl, ul, 32, 0.02, red)


def test_rnnt_edges(binding, oracle_mod):
    # U_b = 0 (blanks only), T_b = 1, and an unusable utterance (label = blank)
    z, labels, tl, ul = _make(9, 4, 8, 3, 11, 10, torch.float32, ragged=False)
    ul[0] = 0
    tl[1] = 1
    labels[2, 0] = 10
    loss, grad = _check(binding, oracle_mod, z, labels, tl, ul, 10, 0.0, "none")
    assert torch.isnan(loss[2]) and not grad[2].any()


def test_rnnt_labels_past_1024(binding, oracle_mod):
    # 1101 lattice rows: the lattice runs as a cluster of bands
    z, labels, tl, ul = _make(5, 1, 260, 1100, 9, 8, torch.float32, ragged=False)
    _check(binding, oracle_mod, z, labels, tl, ul, 8, 0.0, "none")


def test_rnnt_in_place(binding):
    z, labels, tl, ul = _make(3, 3, 20, 7, 64, 63, torch.float32)
    loss, grad = binding.tdt_rnnt_loss_fwd_bwd(z, labels, tl, ul, 63, 0.0, "sum")
    zi = z.clone()
    loss_i, _ = binding.tdt_rnnt_loss_fwd_bwd(zi, labels, tl, ul, 63, 0.0, "sum", grad_out=zi)
    torch.cuda.synchronize()
    assert torch.equal(loss, loss_i) and torch.equal(zi, grad)


def test_rnnt_full_size(binding, oracle_mod):
    # the pages' benchmark size without a duration head, compared in full
    from transducer_loss_asr_gb300.workloads import make_inputs

    inp = make_inputs("parakeet_rnnt", device="cuda")
    _check(binding, oracle_mod, inp["logits"], inp["labels"], inp["logit_lens"],
           inp["label_lens"], inp["blank"], inp["sigma"], inp["reduction"])
