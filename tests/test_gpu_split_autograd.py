"""Split forward/backward API, PyTorch autograd op, torch.compile, in-place
gradient and the data-parallel helper, on the GPU.

* tdt_loss_fwd + tdt_loss_bwd (upstream 1) give the fused call's loss and
  gradient bit for bit (same kernels, x * 1 is exact).
* An upstream gradient g_b scales utterance b's gradient: checked against
  the oracle gradient times g_b within the parity tolerances.
* The autograd op (custom op + fake) passes torch.library.opcheck, and its
  gradient through loss.backward() -- also through a strided view of a wider
  logits tensor -- matches the fused call; torch.compile(fullgraph=True)
  gives the eager results.
* grad_out == logits (contiguous) writes the same gradient over the logits.
"""
import numpy as np
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-6, 1e-5), "f16": (2e-3, 2e-2), "bf16": (2e-3, 2e-2)}


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _inputs(dtype="f32", reduction="mean_volume", base_vd=None, seed=91, B=3):
    w = scaled(WORKLOADS["tiny"], name="split_%s_%s" % (dtype, reduction), B=B, T=23, U=7,
               V=300, blank=299, durations=(0, 1, 2, 3, 4), dtype=dtype, std=1.0, sigma=0.05,
               reduction=reduction, T_range=(11, 23), U_range=(2, 7), base_vd=base_vd,
               seed=seed)
    return make_inputs(w, device="cuda")


def _args(inp):
    return (inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"],
            inp["durations"], inp["blank"])


@pytest.mark.parametrize("dtype,base_vd", [("f32", None), ("bf16", 320), ("f16", None)])
def test_split_equals_fused(binding, dtype, base_vd):
    inp = _inputs(dtype, base_vd=base_vd)
    kw = dict(sigma=inp["sigma"], reduction=inp["reduction"])
    loss_f, grad_f = binding.tdt_loss_fwd_bwd(*_args(inp), **kw)
    loss_s, ws = binding.tdt_loss_fwd(*_args(inp), **kw)
    grad_s = binding.tdt_loss_bwd(*_args(inp), ws, None, **kw)
    torch.cuda.synchronize()
    assert torch.equal(loss_f, loss_s)
    assert torch.equal(grad_f, grad_s)


def test_upstream_gradient_scales_per_utterance(binding, oracle_mod):
    inp = _inputs("f32", reduction="none")
    kw = dict(sigma=inp["sigma"], reduction="none")
    loss, ws = binding.tdt_loss_fwd(*_args(inp), **kw)
    g = torch.tensor([0.25, -1.75, 3.0], dtype=torch.float32, device="cuda")
    grad = binding.tdt_loss_bwd(*_args(inp), ws, g, **kw)
    torch.cuda.synchronize()
    ref = oracle_mod.tdt_loss(inp["logits"].cpu().numpy(), inp["labels"].cpu().numpy(),
                              inp["logit_lens"].cpu().numpy(), inp["label_lens"].cpu().numpy(),
                              inp["durations"], inp["blank"], inp["sigma"], "none")
    np.testing.assert_allclose(loss.double().cpu().numpy(), ref.loss, rtol=1e-6)
    want = ref.grad * g.double().cpu().numpy()[:, None, None, None]
    err = np.abs(grad.double().cpu().numpy() - want).max()
    assert err <= 1e-5 * 3.0, err


@pytest.mark.parametrize("dtype,base_vd,reduction",
                         [("f32", None, "mean_volume"), ("bf16", 320, "none"),
                          ("f32", 311, "mean")])
def test_autograd_matches_fused(binding, dtype, base_vd, reduction):
    from transducer_loss_asr_gb300.autograd import tdt_loss

    inp = _inputs(dtype, reduction=reduction, base_vd=base_vd)
    kw = dict(sigma=inp["sigma"], reduction=reduction)
    loss_f, grad_f = binding.tdt_loss_fwd_bwd(*_args(inp), **kw)
    base = inp["logits"]._base if inp["logits"]._base is not None else inp["logits"]
    leaf = base.detach().clone().requires_grad_(True)
    view = leaf[..., : inp["logits"].shape[-1]] if base_vd else leaf
    loss = tdt_loss(view, inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
                    inp["blank"], inp["sigma"], reduction)
    assert loss.shape == ((inp["logits"].shape[0],) if reduction == "none" else ())
    assert torch.equal(loss.reshape(-1), loss_f.reshape(-1))
    loss.sum().backward()
    g = leaf.grad[..., : inp["logits"].shape[-1]] if base_vd else leaf.grad
    assert torch.equal(g, grad_f)
    if base_vd:  # the columns outside the view get no gradient
        assert not leaf.grad[..., inp["logits"].shape[-1]:].any()


def test_opcheck(binding):
    from transducer_loss_asr_gb300 import autograd  # noqa: F401 (registers the ops)

    inp = _inputs("f32", reduction="mean_volume", B=2)
    logits = inp["logits"].detach().clone().requires_grad_(True)
    args = (logits, inp["labels"], inp["logit_lens"], inp["label_lens"], list(inp["durations"]),
            inp["blank"], inp["sigma"], "mean_volume")
    torch.library.opcheck(torch.ops.tdt_gb300.tdt_loss_forward.default, args)


def test_torch_compile_fullgraph_matches_eager(binding):
    from transducer_loss_asr_gb300.autograd import tdt_loss

    inp = _inputs("bf16", reduction="mean_batch", B=2)

    def f(z):
        return tdt_loss(z, inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
                        inp["blank"], inp["sigma"], "mean_batch") * 2.0

    z1 = inp["logits"].detach().clone().requires_grad_(True)
    z2 = inp["logits"].detach().clone().requires_grad_(True)
    l1 = f(z1)
    l1.backward()
    l2 = torch.compile(f, fullgraph=True)(z2)
    l2.backward()
    assert torch.equal(l1, l2)
    assert torch.equal(z1.grad, z2.grad)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place_gradient(binding, dtype):
    inp = _inputs(dtype, reduction="sum")
    kw = dict(sigma=inp["sigma"], reduction="sum")
    loss_f, grad_f = binding.tdt_loss_fwd_bwd(*_args(inp), **kw)
    z = inp["logits"].clone()
    loss_i, g_i = binding.tdt_loss_fwd_bwd(z, *_args(inp)[1:], grad_out=z, **kw)
    torch.cuda.synchronize()
    assert g_i.data_ptr() == z.data_ptr()
    assert torch.equal(loss_i, loss_f) and torch.equal(z, grad_f)
    # split API: the backward call writes over the logits
    z = inp["logits"].clone()
    loss_s, ws = binding.tdt_loss_fwd(z, *_args(inp)[1:], **kw)
    binding.tdt_loss_bwd(z, *_args(inp)[1:], ws, None, grad_out=z, **kw)
    torch.cuda.synchronize()
    assert torch.equal(z, grad_f)


def test_partial_overlap_rejected(binding):
    inp = _inputs("f32", reduction="sum")
    n = inp["logits"].numel()
    buf = torch.empty(n + 4, dtype=torch.float32, device="cuda")
    z = buf[:n].view(inp["logits"].shape)
    z.copy_(inp["logits"])
    g = buf[4:].view(inp["logits"].shape)  # overlaps the logits, shifted by 4 elements
    with pytest.raises(binding.TDTError) as e:
        binding.tdt_loss_fwd_bwd(z, *_args(inp)[1:], sigma=inp["sigma"], reduction="sum",
                                 grad_out=g)
    assert e.value.status == -13


def test_sharded_single_rank_equals_fused(binding):
    from transducer_loss_asr_gb300.sharding import sharded_tdt_loss

    for red in ("mean_volume", "none"):
        inp = _inputs("f32", reduction=red)
        kw = dict(sigma=inp["sigma"], reduction=red)
        loss_f, grad_f = binding.tdt_loss_fwd_bwd(*_args(inp), **kw)
        loss_s, grad_s = sharded_tdt_loss(*_args(inp), **kw)
        torch.cuda.synchronize()
        np.testing.assert_allclose(loss_s.double().cpu().numpy().reshape(-1),
                                   loss_f.double().cpu().numpy().reshape(-1), rtol=1e-6)
        assert torch.equal(grad_s, grad_f)
