"""GPU (C ABI) versus the CPU oracle, element by element.

Tolerances (fp32 logits): loss relative error <= 1e-6, gradient absolute
error <= 1e-5.  bf16/fp16 logits: loss relative <= 2e-3, gradient absolute
<= 2e-2, against the oracle run on the same up-cast inputs; bf16/fp16 are
also held to a tighter bound, one unit in the last place of the stored
gradient plus 2e-6, since the kernels compute in fp32 and round once.
"""
import numpy as np
import pytest
import torch

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-6, 1e-5), "f16": (2e-3, 2e-2), "bf16": (2e-3, 2e-2)}
ULP = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def run_gpu(binding, inp, compute_grad=True):
    loss, grad = binding.tdt_loss_fwd_bwd(
        inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
        inp["blank"], inp["sigma"], inp["reduction"], compute_grad=compute_grad)
    torch.cuda.synchronize()
    return loss, grad


def run_oracle(oracle_mod, inp, rows=None, want_grad=True):
    return oracle_mod.tdt_loss(
        inp["logits"].float().cpu().numpy(), inp["labels"].cpu().numpy(),
        inp["logit_lens"].cpu().numpy(), inp["label_lens"].cpu().numpy(), inp["durations"],
        inp["blank"], inp["sigma"], inp["reduction"], want_grad=want_grad, rows=rows)


def check_loss(l_gpu, l_ref, dtype, margin=None):
    """Loss relative error within the dtype's tolerance; NaN and +inf where
    the oracle has them.  margin(quantity, error, tolerance) records it."""
    rtol = TOL[dtype][0]
    l_gpu = l_gpu.double().cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isnan(l_gpu), np.isnan(l_ref))
    assert np.array_equal(np.isposinf(l_gpu), np.isposinf(l_ref))
    rel = np.abs(l_gpu[fin] - l_ref[fin]) / np.maximum(np.abs(l_ref[fin]), 1e-30)
    worst = float(rel.max()) if rel.size else 0.0
    if margin:
        margin("loss_rel", worst, rtol)
    assert worst <= rtol, "loss rel err %.3e > %.1e" % (worst, rtol)
    return worst


def check_grad(g_gpu, g_ref, dtype, chunk=1 << 24, margin=None):
    """Every element: absolute error within the dtype's tolerance (and, for
    16-bit dtypes, within one ulp of the stored value plus 2e-6).  Compared
    in chunks of the flattened arrays to bound host memory."""
    atol = TOL[dtype][1]
    g_flat = g_gpu.reshape(-1)
    r_flat = g_ref.reshape(-1)
    assert g_flat.numel() == r_flat.size
    worst = 0.0
    worst_ulp = 0.0
    for s in range(0, r_flat.size, chunk):
        g = g_flat[s:s + chunk].double().cpu().numpy()
        r = r_flat[s:s + chunk]
        err = np.abs(g - r)
        if not err.size:
            continue
        worst = max(worst, float(err.max()))
        assert err.max() <= atol, "grad abs err %.3e > %.1e" % (err.max(), atol)
        if dtype in ULP:
            bound = np.abs(r) * ULP[dtype] + 2e-6
            worst_ulp = max(worst_ulp, float((err / bound).max()))
            assert (err <= bound).all(), "grad beyond one ulp: %.3e" % (err - bound).max()
    if margin:
        margin("grad_abs", worst, atol)
        if dtype in ULP:
            margin("grad_ulp", worst_ulp, 1.0)
    return worst


def full_check(binding, oracle_mod, inp, record_margin=None, case=None):
    w = inp["workload"]
    margin = None
    if record_margin is not None:
        name = case or w.name

        def margin(q, e, t):
            return record_margin(name, q, e, t)
    loss, grad = run_gpu(binding, inp)
    ref = run_oracle(oracle_mod, inp)
    check_loss(loss, ref.loss, w.dtype, margin)
    check_grad(grad, ref.grad, w.dtype, margin=margin)
    return loss, grad, ref


# ------------------------------------------------------------- small and medium

def test_tiny_workload(binding, oracle_mod, record_margin):
    full_check(binding, oracle_mod, make_inputs("tiny", device="cuda"), record_margin)


MEDIUM = {
    # several warp tiles per row, a ragged tail (V not a multiple of 256), ragged lengths
    "f32_ragged_view": dict(B=3, T=37, U=11, V=1000, blank=999, durations=(0, 1, 2, 3, 4),
                            dtype="f32", std=1.0, sigma=0.05, reduction="mean_volume",
                            T_range=(20, 37), U_range=(3, 11), base_vd=1013),
    "bf16_ragged_view": dict(B=4, T=29, U=9, V=777, blank=776, durations=(0, 1, 2, 3),
                             dtype="bf16", std=1.5, sigma=0.1, reduction="mean",
                             T_range=(10, 29), U_range=(1, 9), base_vd=790),
    "f16_full": dict(B=2, T=18, U=6, V=513, blank=512, durations=(0, 1, 2), dtype="f16",
                     std=1.0, sigma=0.0, reduction="sum"),
    # strided views whose rows sit at varying offsets from the gradient rows'
    # 16-byte boundaries (the realigned vector path), short and long rows
    "f16_ragged_view": dict(B=3, T=21, U=7, V=555, blank=554, durations=(0, 1, 2, 3, 4),
                            dtype="f16", std=1.0, sigma=0.05, reduction="mean_volume",
                            T_range=(9, 21), U_range=(2, 7), base_vd=571),
    "bf16_short_view": dict(B=3, T=17, U=5, V=45, blank=44, durations=(0, 1, 2),
                            dtype="bf16", std=1.0, sigma=0.0, reduction="sum",
                            T_range=(8, 17), U_range=(1, 5), base_vd=61),
    "f32_short_view": dict(B=2, T=13, U=4, V=37, blank=36, durations=(0, 2, 3), dtype="f32",
                           std=1.0, sigma=0.02, reduction="mean_batch", T_range=(6, 13),
                           U_range=(1, 4), base_vd=50),
    "f32_no_zero_duration": dict(B=2, T=25, U=5, V=64, blank=63, durations=(1, 2, 4),
                                 dtype="f32", std=2.0, sigma=0.02, reduction="none",
                                 T_range=(12, 25), U_range=(0, 5)),
    "f32_unsorted_blank_first": dict(B=3, T=15, U=4, V=40, blank=0, durations=(3, 0, 1),
                                     dtype="f32", std=1.0, sigma=0.0, reduction="mean_batch"),
    "f32_long_rows": dict(B=1, T=9, U=3, V=20001, blank=20000, durations=(0, 1, 2, 3, 4),
                          dtype="f32", std=1.0, sigma=0.0, reduction="sum"),
    "f32_many_durations": dict(B=2, T=40, U=8, V=33, blank=32, durations=tuple(range(17)),
                               dtype="f32", std=1.0, sigma=0.3, reduction="mean_volume"),
    "f32_labels_past_1024": dict(B=1, T=300, U=1100, V=9, blank=8, durations=(0, 1, 2),
                                 dtype="f32", std=1.0, sigma=0.0, reduction="none"),
}


@pytest.mark.parametrize("name", sorted(MEDIUM))
def test_medium_cases(binding, oracle_mod, record_margin, name):
    w = scaled(WORKLOADS["tiny"], name=name, seed=777, **MEDIUM[name])
    full_check(binding, oracle_mod, make_inputs(w, device="cuda"), record_margin)


# Problems whose logits reach 8 MiB go through the chunked multi-stream
# schedule (up to four chunks of utterances); smaller ones run serially on the
# caller's stream.  These cases sit above that size: B=5 splits unevenly into
# chunks of 1,1,1,2 utterances, B=2 into two chunks and B=1 into one.  The
# tall ragged case has lattices too tall for one CTA, so each chunk's
# lattice runs as bands exchanging boundary rows through global memory
# beside the other chunks' passes, some bands wholly above U_b.
CHUNKED = {
    "f32_b5_ragged_view": dict(B=5, T=24, U=6, V=8193, blank=8192, durations=(0, 1, 2, 3, 4),
                               dtype="f32", std=1.0, sigma=0.05, reduction="mean_volume",
                               T_range=(12, 24), U_range=(2, 6), base_vd=8203),
    "bf16_b4_ragged_view": dict(B=4, T=30, U=8, V=8193, blank=8192, durations=(0, 1, 2, 3),
                                dtype="bf16", std=1.5, sigma=0.0, reduction="mean_batch",
                                T_range=(15, 30), U_range=(1, 8), base_vd=8205),
    "f16_b2_full": dict(B=2, T=30, U=8, V=16001, blank=16000, durations=(0, 1, 2),
                        dtype="f16", std=1.0, sigma=0.02, reduction="sum"),
    "f32_b1_full": dict(B=1, T=50, U=10, V=4097, blank=4096, durations=(0, 1, 2, 3, 4),
                        dtype="f32", std=1.0, sigma=0.0, reduction="none"),
    "f32_b3_tall_ragged": dict(B=3, T=40, U=700, V=30, blank=29, durations=(0, 1, 2),
                               dtype="f32", std=1.0, sigma=0.02, reduction="none",
                               T_range=(20, 40), U_range=(300, 700)),
}


@pytest.mark.parametrize("name", sorted(CHUNKED))
def test_chunked_schedule_cases(binding, oracle_mod, record_margin, name):
    w = scaled(WORKLOADS["tiny"], name=name, seed=919, **CHUNKED[name])
    esize = 4 if w.dtype == "f32" else 2
    assert w.B * w.T * (w.U + 1) * w.VD * esize >= 8 << 20
    full_check(binding, oracle_mod, make_inputs(w, device="cuda"), record_margin)


@pytest.mark.parametrize("red", ["none", "sum", "mean", "mean_batch", "mean_volume"])
def test_every_reduction(binding, oracle_mod, red):
    w = scaled(WORKLOADS["tiny"], name="red_" + red, B=5, T=14, U=5, V=50, blank=49,
               durations=(0, 1, 2), sigma=0.05, reduction=red, T_range=(6, 14), U_range=(1, 5),
               seed=31)
    full_check(binding, oracle_mod, make_inputs(w, device="cuda"))


# ------------------------------------------------------------- edge cases

def test_empty_batch(binding):
    for red, expect in (("sum", 0.0), ("mean_batch", np.nan), ("none", None)):
        z = torch.zeros(0, 5, 3, 10, device="cuda")
        e = torch.zeros(0, dtype=torch.int64, device="cuda")
        loss, grad = binding.tdt_loss_fwd_bwd(z, torch.zeros(0, 2, dtype=torch.int64,
                                                             device="cuda"), e, e, [0, 1, 2], 6,
                                              0.0, red)
        torch.cuda.synchronize()
        if expect is None:
            assert loss.numel() == 0
        elif np.isnan(expect):
            assert torch.isnan(loss).all()
        else:
            assert loss.item() == expect
        assert grad.numel() == 0


def test_no_labels_at_all(binding, oracle_mod):
    w = scaled(WORKLOADS["tiny"], name="no_labels", U=0, T=11, durations=(0, 1, 2),
               V=7, blank=6, reduction="sum", seed=5)
    full_check(binding, oracle_mod, make_inputs(w, device="cuda"))


def test_degenerate_utterances(binding, oracle_mod):
    """No path (+inf, zero rows), unusable lengths/labels (NaN, zero rows),
    T_b = 1, U_b = 0, durations longer than the utterance."""
    w = scaled(WORKLOADS["tiny"], name="degenerate", B=6, T=9, U=3, V=6, blank=5,
               durations=(0, 2, 11), reduction="none", seed=8)
    inp = make_inputs(w, device="cuda")
    inp["logit_lens"] = torch.tensor([9, 8, 1, 9, 12, 4], device="cuda")   # 9 odd: no path
    inp["label_lens"] = torch.tensor([3, 2, 0, 0, 1, 2], device="cuda")
    labels = inp["labels"].clone()
    labels[:, :] = 1
    labels[1, 2:] = -100
    labels[2, :] = -100
    labels[3, :] = -100
    labels[4, 1:] = -100
    labels[5, 1] = 5     # blank used as a label -> unusable
    labels[5, 2:] = -100
    inp["labels"] = labels
    loss, grad, ref = full_check(binding, oracle_mod, inp)
    l = loss.cpu().numpy()
    assert np.isposinf(l[0]) and np.isnan(l[4]) and np.isnan(l[5])
    g = grad.cpu()
    assert (g[0] == 0).all() and (g[4] == 0).all() and (g[5] == 0).all()


def test_loss_only_matches(binding, oracle_mod):
    inp = make_inputs(scaled(WORKLOADS["parakeet_bf16_ragged"], B=3, T=30, U=6, V=301,
                             blank=300, base_vd=320, T_range=(12, 30), U_range=(2, 6)),
                      device="cuda")
    l1, g1 = run_gpu(binding, inp, compute_grad=False)
    assert g1 is None
    l2, g2 = run_gpu(binding, inp)
    assert torch.equal(l1, l2)
    ref = run_oracle(oracle_mod, inp, want_grad=False)
    check_loss(l1, ref.loss, "bf16")


def test_workspace_variant_and_determinism(binding):
    inp = make_inputs(scaled(WORKLOADS["parakeet"], B=2, T=40, U=9, V=2049, blank=2048),
                      device="cuda")
    l1, g1 = run_gpu(binding, inp)
    need = binding.tdt_loss_workspace_size(inp["logits"].shape, len(inp["durations"]))
    ws = torch.full((need,), 0x7f, dtype=torch.uint8, device="cuda")
    l2, g2 = binding.tdt_loss_fwd_bwd_ws(
        inp["logits"], inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
        inp["blank"], ws, inp["sigma"], inp["reduction"])
    torch.cuda.synchronize()
    assert torch.equal(l1, l2) and torch.equal(g1, g2)
    l3, g3 = run_gpu(binding, inp)
    assert torch.equal(l1, l3) and torch.equal(g1, g3)


def test_closed_form_long_lattice(binding, oracle_mod, record_margin):
    """Uniform logits, durations [0, 1], T = 900, U = 1200: the exact loss is a
    log-sum of binomial terms; pins the long fixed-point lattice on the GPU.
    The gradient is compared with the oracle's at every element."""
    from scipy.special import gammaln, logsumexp

    T, U, V, sigma = 900, 1200, 4, 0.02
    z = torch.zeros(1, T, U + 1, V + 2, device="cuda")
    labels = torch.zeros(1, U, dtype=torch.int64, device="cuda")
    tl = torch.tensor([T], device="cuda")
    ul = torch.tensor([U], device="cuda")
    loss, grad = binding.tdt_loss_fwd_bwd(z, labels, tl, ul, [0, 1], V - 1, sigma, "none")
    torch.cuda.synchronize()
    c = -np.log(V) - np.log(2) - sigma
    ks = np.arange(0, min(U, T - 1) + 1)
    terms = (gammaln(U + 1) - gammaln(ks + 1) - gammaln(U - ks + 1)
             + gammaln(U + T - ks) - gammaln(U + 1) - gammaln(T - ks) + (U + T - ks) * c)
    expect = -logsumexp(terms)
    rel = abs(loss.item() - expect) / expect
    record_margin("closed_form_T900_U1200", "loss_rel_closed_form", rel, 1e-6)
    assert rel <= 1e-6
    ref = oracle_mod.tdt_loss(z.cpu().numpy(), labels.cpu().numpy(), tl.cpu().numpy(),
                              ul.cpu().numpy(), [0, 1], V - 1, sigma, "none")
    assert abs(ref.loss[0] - expect) / expect <= 1e-9
    check_loss(loss, ref.loss, "f32",
               lambda q, e, t: record_margin("closed_form_T900_U1200", q, e, t))
    check_grad(grad, ref.grad, "f32",
               margin=lambda q, e, t: record_margin("closed_form_T900_U1200", q, e, t))


# ------------------------------------------------------------- full-size workloads

def _padding_rows_are_zero(grad_b, Tb, Ub):
    """Rows outside the lattice of one utterance (t >= T_b or u > U_b) hold
    exact zeros."""
    T, U1 = grad_b.shape[0], grad_b.shape[1]
    t = torch.arange(T, device=grad_b.device)[:, None]
    u = torch.arange(U1, device=grad_b.device)[None, :]
    pad = (t >= Tb) | (u > Ub)
    return bool((grad_b[pad] == 0).all().item())


@pytest.mark.parametrize("name", ["parakeet", "parakeet_bf16_ragged"])
def test_full_size_parakeet(binding, oracle_mod, record_margin, name):
    inp = make_inputs(name, device="cuda")
    base = inp["logits"]._base if inp["logits"]._base is not None else inp["logits"]
    before = base.float().sum().item()
    _, grad, _ = full_check(binding, oracle_mod, inp, record_margin)
    assert base.float().sum().item() == before   # the input (and its wider base) is untouched
    tl, ul = inp["logit_lens"].tolist(), inp["label_lens"].tolist()
    for b in range(grad.shape[0]):
        assert _padding_rows_are_zero(grad[b], tl[b], ul[b])


def test_full_size_large_batch_every_row(binding, oracle_mod, record_margin):
    """B16 T750 U120 V1025 bf16, ragged: every gradient element of every
    utterance against the oracle.  The reduction is sum, so c_b = 1 and the
    rows of utterance b equal those of a batch holding b alone: the oracle
    runs one utterance at a time, which bounds its float64 memory."""
    inp = make_inputs("large_batch", device="cuda")
    w = inp["workload"]
    assert w.reduction == "sum"
    loss, grad = run_gpu(binding, inp)

    def margin(q, e, t):
        return record_margin(w.name, q, e, t)

    tl, ul = inp["logit_lens"].tolist(), inp["label_lens"].tolist()
    total = 0.0
    for b in range(w.B):
        sub = dict(inp)
        for k in ("logits", "labels", "logit_lens", "label_lens"):
            sub[k] = inp[k][b:b + 1]
        ref = run_oracle(oracle_mod, sub)
        total += float(ref.loss[0])
        check_grad(grad[b], ref.grad[0], w.dtype, margin=margin)
        assert _padding_rows_are_zero(grad[b], tl[b], ul[b])
    check_loss(loss, np.array([total]), w.dtype, margin)


def test_full_size_long_labels_every_row(binding, oracle_mod, record_margin):
    """B1 T2000 U1200 V129 D9 fp32, sigma 0.02: every one of the 331,476,000
    gradient elements against the float64 oracle at the fp32 tolerances --
    the longest lattice (3,200 anti-diagonals) of the five workloads."""
    inp = make_inputs("long_labels", device="cuda")
    full_check(binding, oracle_mod, inp, record_margin)


# ------------------------------------------------------------- lattice bands

BANDED = {
    "d5_ragged": dict(B=3, T=37, U=40, V=100, blank=99, durations=(0, 1, 2, 3, 4), dtype="f32",
                      std=1.0, sigma=0.05, reduction="mean_volume", T_range=(20, 37),
                      U_range=(25, 40)),
    "d9_long": dict(B=2, T=60, U=70, V=50, blank=49, durations=tuple(range(9)), dtype="f32",
                    std=1.0, sigma=0.02, reduction="none"),
    "d3_no_zero": dict(B=2, T=45, U=33, V=40, blank=0, durations=(1, 2, 4), dtype="bf16",
                       std=1.5, sigma=0.0, reduction="sum", T_range=(30, 45), U_range=(5, 33)),
}


@pytest.mark.parametrize("name", sorted(BANDED))
def test_lattice_bands_do_not_change_results(binding, oracle_mod, record_margin, name):
    """The lattice rows are split into K bands (one CTA each) that exchange
    boundary rows in a thread-block cluster (exchange 1) or through global
    memory (exchange 2); the arithmetic per node is the same for every K and
    either exchange, so the loss and the gradient must agree bit for bit, and
    with the oracle."""
    w = scaled(WORKLOADS["tiny"], name="bands_" + name, seed=4242, **BANDED[name])
    inp = make_inputs(w, device="cuda")
    results = []
    cases = [(K, 0) for K in (0, 1, 2, 3, 7, 16)] + [(K, 2) for K in (2, 3, 7, 24, 80)]
    for K, mode in cases:
        prev = binding.tdt_loss_set_lattice_bands(K)
        prev_mode = binding.tdt_loss_set_lattice_exchange(mode)
        try:
            loss, grad = run_gpu(binding, inp)
        finally:
            binding.tdt_loss_set_lattice_bands(prev)
            binding.tdt_loss_set_lattice_exchange(prev_mode)
        results.append(((K, mode), loss.clone(), grad.clone()))
    for case, loss, grad in results[1:]:
        assert torch.equal(loss, results[0][1]), "loss differs with bands/exchange %s" % (case,)
        assert torch.equal(grad, results[0][2]), "grad differs with bands/exchange %s" % (case,)
    ref = run_oracle(oracle_mod, inp)

    def margin(q, e, t):
        return record_margin("bands_" + name, q, e, t)
    check_loss(results[0][1], ref.loss, w.dtype, margin)
    check_grad(results[0][2], ref.grad, w.dtype, margin=margin)


# ------------------------------------------------------------- CUDA graphs

@pytest.mark.parametrize("seed", range(12))
def test_global_bands_match_one_band_on_random_shapes(binding, seed):
    """Bands exchanging boundary rows through global memory compute every
    node with the same arithmetic as one band, so on random shapes (ragged
    lengths, random duration sets with and without 0, fp32 and bf16) any
    band count must reproduce bit for bit the result with one band forced
    (or the fewest cluster bands whose rings fit, for lattices one CTA cannot
    hold).  Up to 80 bands for up to three utterances is more CTAs than the
    GPU holds at once: the start-order tickets keep every wait on a CTA that
    has started."""
    rng = np.random.default_rng(9000 + seed)
    T = int(rng.integers(5, 60))
    U = int(rng.integers(20, 200))
    V = int(rng.integers(20, 60))
    nd = int(rng.integers(1, 10))
    durs = sorted(int(d) for d in rng.choice(np.arange(0, 9), size=nd, replace=False))
    if max(durs) == 0:
        durs = [0, 1]
    B = int(rng.integers(1, 4))
    dtype = "f32" if seed % 3 else "bf16"
    w = scaled(WORKLOADS["tiny"], name="gxr%d" % seed, B=B, T=T, U=U, V=V, blank=V - 1,
               durations=tuple(durs), dtype=dtype, std=1.0, sigma=0.02, reduction="none",
               T_range=(max(1, T // 2), T), U_range=(U // 2, U), seed=5150 + seed)
    inp = make_inputs(w, device="cuda")
    K = int(rng.integers(2, min(80, U + 1) + 1))
    results = []
    for bands, mode in ((1, 0), (K, 2)):
        prev = binding.tdt_loss_set_lattice_bands(bands)
        prev_mode = binding.tdt_loss_set_lattice_exchange(mode)
        try:
            loss, grad = run_gpu(binding, inp)
        finally:
            binding.tdt_loss_set_lattice_bands(prev)
            binding.tdt_loss_set_lattice_exchange(prev_mode)
        results.append((loss.clone(), grad.clone()))
    assert torch.equal(results[0][0], results[1][0]), "loss differs with %d global bands" % K
    assert torch.equal(results[0][1], results[1][1]), "grad differs with %d global bands" % K


GRAPH_SHAPES = {
    "serial": dict(V=200, U=6, U_range=(2, 6)),
    "chunked": dict(V=8193, U=6, U_range=(2, 6)),
    # lattices too tall for one CTA: bands exchanging boundary rows through
    # global memory, with their start-order counters and polls, inside the
    # captured graph (one launch for the batch, and one per chunk)
    "tall_serial": dict(V=20, U=600, U_range=(300, 600)),
    "tall_chunked": dict(V=60, U=600, U_range=(300, 600)),
}


@pytest.mark.parametrize("shape", sorted(GRAPH_SHAPES))
@pytest.mark.parametrize("own_workspace", [True, False])
def test_cuda_graph_capture_and_replay(binding, own_workspace, shape):
    """The call is stream-ordered (small problems run on the caller's stream;
    larger ones fork internal streams from it and join them back through
    events), so it can be captured into a CUDA graph; replays give the eager
    results, also after the inputs change in place.  V=8193 (and the tall
    case with V=60) put the logits above the 8 MiB size of the chunked
    schedule."""
    g = GRAPH_SHAPES[shape]
    w = scaled(WORKLOADS["tiny"], name="graph", B=3, T=21, U=g["U"], V=g["V"], blank=g["V"] - 1,
               durations=(0, 1, 2, 3, 4), sigma=0.05, reduction="mean_volume",
               T_range=(10, 21), U_range=g["U_range"], seed=606)
    esize = 4
    chunked = w.B * w.T * (w.U + 1) * w.VD * esize >= 8 << 20
    assert chunked == shape.endswith("chunked")
    inp = make_inputs(w, device="cuda")
    z = inp["logits"]
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(z)
    ws = torch.empty(binding.workspace_size(z.shape, len(inp["durations"])), dtype=torch.uint8,
                     device="cuda")
    args = (z, inp["labels"], inp["logit_lens"], inp["label_lens"], inp["durations"],
            inp["blank"])

    def call():
        if own_workspace:
            binding.tdt_loss_fwd_bwd_ws(*args, ws, sigma=inp["sigma"], reduction="mean_volume",
                                        loss_out=loss, grad_out=grad)
        else:
            binding.tdt_loss_fwd_bwd(*args, inp["sigma"], "mean_volume", loss_out=loss,
                                     grad_out=grad)

    call()  # eager first: creates the library's streams and sets kernel attributes
    torch.cuda.synchronize()
    ref_loss, ref_grad = loss.clone(), grad.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    loss.zero_()
    grad.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(loss, ref_loss) and torch.equal(grad, ref_grad)
    # new values in the captured input buffer: the replay computes them
    z.mul_(1.5)
    call()
    torch.cuda.synchronize()
    eager_loss, eager_grad = loss.clone(), grad.clone()
    loss.zero_()
    grad.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(loss, eager_loss) and torch.equal(grad, eager_grad)
    assert not torch.equal(eager_loss, ref_loss)
