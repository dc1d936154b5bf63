"""Pins of the CPU oracle against things other than itself (no GPU needed).

* brute-force enumeration of every alignment path (the definition of the loss),
* the lattice path sum through a linear solve of (I - M) (alpha and beta at
  every node, without the recursion),
* closed forms for uniform logits,
* central finite differences of the float64 loss (the gradient),
* invariants that hold for any input,
* log-softmax tables against scipy's log_softmax.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import gammaln, log_softmax, logsumexp

from lattice_pins import enumerate_paths, node_log_probs, path_sum_linear
from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs


def _np_inputs(name="tiny", **over):
    inp = make_inputs(name)
    z = inp["logits"].float().numpy()
    return (z, inp["labels"].numpy(), inp["logit_lens"].numpy(), inp["label_lens"].numpy(),
            inp["workload"])


def _random_case(rng, B, T, U, V, durations, blank=None, sigma=0.0, ragged=False, std=1.5,
                 extra_vd=0):
    D = len(durations)
    base = rng.normal(0.0, std, size=(B, T, U + 1, V + D + extra_vd))
    z = base[..., : V + D] if extra_vd else base
    if blank is None:
        blank = V - 1
    toks = [k for k in range(V) if k != blank]
    labels = rng.choice(toks, size=(B, max(U, 1))).astype(np.int64)
    if ragged:
        tl = rng.integers(1, T + 1, size=B).astype(np.int64)
        ul = rng.integers(0, U + 1, size=B).astype(np.int64)
    else:
        tl = np.full(B, T, dtype=np.int64)
        ul = np.full(B, U, dtype=np.int64)
    for b in range(B):
        labels[b, ul[b]:] = -100
    return z, labels, tl, ul, blank


# ---------------------------------------------------------------- brute force

def test_tiny_workload_matches_path_enumeration(oracle_mod):
    """The tiny workload (B2 T12 U4 V9, durations 0..3): every alignment path."""
    z, labels, tl, ul, w = _np_inputs("tiny")
    r = oracle_mod.tdt_loss(z, labels, tl, ul, w.durations, w.blank, w.sigma, "none",
                            want_grad=False)
    for b in range(w.B):
        lpb, lpl, lpd = node_log_probs(z[b].astype(np.float64), w.V, w.blank, labels[b], w.T, w.U)
        ll, n_paths = enumerate_paths(lpb, lpl, lpd, w.T, w.U, w.durations, w.sigma)
        assert n_paths == 2028199
        assert r.utt_loss[b] == pytest.approx(-ll, rel=1e-12)


@pytest.mark.parametrize("case", range(8))
def test_random_lattices_match_path_enumeration(oracle_mod, case):
    """Random small lattices: sigma > 0, ragged lengths, durations without 0,
    non-contiguous durations, blank not last, empty label sequences, a strided
    slice of a wider tensor, float64 and float32 inputs."""
    rng = np.random.default_rng(1000 + case)
    variants = [
        dict(durations=[0, 1, 2], V=5, sigma=0.3),
        dict(durations=[1, 2, 4], V=4, sigma=0.0),
        dict(durations=[0, 2, 3], V=6, sigma=0.1, blank=0),
        dict(durations=[2, 0, 1], V=3, sigma=0.05),            # unsorted
        dict(durations=[1], V=4, sigma=0.2),
        dict(durations=[0, 1, 2, 3, 4], V=5, sigma=0.0, extra_vd=3),
        dict(durations=[0, 1], V=7, sigma=0.5, blank=3),
        dict(durations=[0, 3], V=4, sigma=0.0),
    ]
    v = variants[case]
    T, U, B = 7, 3, 3
    z, labels, tl, ul, blank = _random_case(rng, B, T, U, v["V"], v["durations"],
                                            blank=v.get("blank"), sigma=v["sigma"],
                                            ragged=True, extra_vd=v.get("extra_vd", 0))
    z32 = z.astype(np.float32)
    for zz in (z, z32):
        r = oracle_mod.tdt_loss(zz, labels, tl, ul, v["durations"], blank, v["sigma"], "none",
                                want_grad=False, want_lattice=True)
        for b in range(B):
            Tb, Ub = int(tl[b]), int(ul[b])
            lpb, lpl, lpd = node_log_probs(np.asarray(zz[b], dtype=np.float64), v["V"], blank,
                                           labels[b], Tb, Ub)
            ll, _ = enumerate_paths(lpb, lpl, lpd, Tb, Ub, v["durations"], v["sigma"])
            if ll == -np.inf:
                assert r.utt_loss[b] == np.inf
            else:
                assert r.utt_loss[b] == pytest.approx(-ll, rel=1e-12, abs=1e-12)
            # alpha / beta at every node against the linear-system path sums
            lz, lF, lG = path_sum_linear(lpb, lpl, lpd, Tb, Ub, v["durations"], v["sigma"])
            a = r.alpha[b, :Tb, : Ub + 1]
            bt = r.beta[b, :Tb, : Ub + 1]
            fin = np.isfinite(lF)
            assert np.array_equal(fin, np.isfinite(a))
            np.testing.assert_allclose(a[fin], lF[fin], rtol=0, atol=1e-9)
            fin = np.isfinite(lG)
            assert np.array_equal(fin, np.isfinite(bt))
            np.testing.assert_allclose(bt[fin], lG[fin], rtol=0, atol=1e-9)


def test_tiny_alpha_beta_match_linear_system(oracle_mod):
    z, labels, tl, ul, w = _np_inputs("tiny")
    r = oracle_mod.tdt_loss(z, labels, tl, ul, w.durations, w.blank, 0.0, "none",
                            want_grad=False, want_lattice=True)
    for b in range(w.B):
        lpb, lpl, lpd = node_log_probs(z[b].astype(np.float64), w.V, w.blank, labels[b], w.T, w.U)
        lz, lF, lG = path_sum_linear(lpb, lpl, lpd, w.T, w.U, w.durations)
        np.testing.assert_allclose(r.alpha[b], lF, rtol=0, atol=1e-10)
        np.testing.assert_allclose(r.beta[b], lG, rtol=0, atol=1e-10)
        assert r.ll_alpha[b] == pytest.approx(lz, abs=1e-10)


# ---------------------------------------------------------------- closed forms

def _uniform_case(T, U, V, D):
    z = np.zeros((1, T, U + 1, V + D), dtype=np.float32)
    labels = np.zeros((1, max(U, 1)), dtype=np.int64)  # label 0, blank = V-1
    return z, labels, np.array([T]), np.array([U])


@pytest.mark.parametrize("T,U,V,sigma", [(5, 2, 3, 0.0), (40, 17, 11, 0.25), (600, 300, 5, 0.02)])
def test_closed_form_single_frame_durations(oracle_mod, T, U, V, sigma):
    """durations = [1], uniform logits: every arc consumes one frame, the last
    is blank, so L = T (log V + sigma) - log C(T-1, U)."""
    z, labels, tl, ul = _uniform_case(T, U, V, 1)
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [1], V - 1, sigma, "none", want_grad=False)
    log_binom = gammaln(T) - gammaln(U + 1) - gammaln(T - U)
    expect = T * (math.log(V) + sigma) - log_binom
    assert r.utt_loss[0] == pytest.approx(expect, rel=1e-12)


@pytest.mark.parametrize("T,U,V,sigma", [(4, 3, 2, 0.0), (30, 12, 7, 0.1), (900, 1200, 4, 0.02)])
def test_closed_form_zero_one_durations(oracle_mod, T, U, V, sigma):
    """durations = [0, 1], uniform logits: with k of the U labels taking d = 1,
    a path has U + T - k arcs of weight c = -log V - log 2 - sigma and there are
    C(U, k) C(U + T - k - 1, U) of them (the last arc is the final blank)."""
    z, labels, tl, ul = _uniform_case(T, U, V, 2)
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [0, 1], V - 1, sigma, "none", want_grad=False)
    c = -math.log(V) - math.log(2) - sigma
    ks = np.arange(0, min(U, T - 1) + 1)
    terms = (gammaln(U + 1) - gammaln(ks + 1) - gammaln(U - ks + 1)
             + gammaln(U + T - ks) - gammaln(U + 1) - gammaln(T - ks) + (U + T - ks) * c)
    expect = -logsumexp(terms)
    assert r.utt_loss[0] == pytest.approx(expect, rel=1e-12)


# ---------------------------------------------------------------- gradients

def _fd_grad(oracle_mod, z, labels, tl, ul, durs, blank, sigma, red, h=1e-5, idx=None):
    flat = z.reshape(-1)
    g = np.zeros_like(flat)
    ids = range(flat.size) if idx is None else idx
    for j in ids:
        old = flat[j]
        flat[j] = old + h
        lp = oracle_mod.tdt_loss(z, labels, tl, ul, durs, blank, sigma, red, want_grad=False).loss.sum()
        flat[j] = old - h
        lm = oracle_mod.tdt_loss(z, labels, tl, ul, durs, blank, sigma, red, want_grad=False).loss.sum()
        flat[j] = old
        g[j] = (lp - lm) / (2 * h)
    return g.reshape(z.shape)


def test_tiny_gradient_matches_finite_differences(oracle_mod):
    """All 1,560 logits of the tiny workload (reduction none = grad of sum L_b)."""
    z, labels, tl, ul, w = _np_inputs("tiny")
    z = z.astype(np.float64)
    r = oracle_mod.tdt_loss(z, labels, tl, ul, w.durations, w.blank, w.sigma, "none")
    fd = _fd_grad(oracle_mod, z.copy(), labels, tl, ul, w.durations, w.blank, w.sigma, "none")
    np.testing.assert_allclose(r.grad, fd, rtol=0, atol=2e-7)


@pytest.mark.parametrize("red", ["none", "sum", "mean", "mean_batch", "mean_volume"])
def test_reduced_gradients_match_finite_differences(oracle_mod, red):
    """Ragged lengths, sigma > 0, a strided input: every reduction's gradient."""
    rng = np.random.default_rng(7)
    z, labels, tl, ul, blank = _random_case(rng, 3, 6, 3, 5, [0, 1, 2], sigma=0.2, ragged=False,
                                            extra_vd=2)
    tl = np.array([6, 4, 5]); ul = np.array([3, 1, 2])
    for b in range(3):
        labels[b, ul[b]:] = -100
    z = np.ascontiguousarray(z)
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [0, 1, 2], blank, 0.2, red)
    fd = _fd_grad(oracle_mod, z.copy(), labels, tl, ul, [0, 1, 2], blank, 0.2, red)
    np.testing.assert_allclose(r.grad, fd, rtol=0, atol=2e-7)
    # rows outside each utterance's lattice are exactly zero
    for b in range(3):
        assert not r.grad[b, tl[b]:].any()
        assert not r.grad[b, :, ul[b] + 1:].any()


def test_reduction_values(oracle_mod):
    rng = np.random.default_rng(11)
    z, labels, tl, ul, blank = _random_case(rng, 4, 6, 3, 5, [0, 1, 2], ragged=True)
    ul = np.maximum(ul, 1)
    for b in range(4):
        labels[b, : ul[b]] = rng.integers(0, blank, size=ul[b])
        labels[b, ul[b]:] = -100
    L = oracle_mod.tdt_loss(z, labels, tl, ul, [0, 1, 2], blank, 0.0, "none", want_grad=False).loss
    get = lambda red: oracle_mod.tdt_loss(z, labels, tl, ul, [0, 1, 2], blank, 0.0, red,
                                          want_grad=False).loss[0]
    assert get("sum") == pytest.approx(L.sum(), rel=1e-14)
    assert get("mean_batch") == pytest.approx(L.mean(), rel=1e-14)
    assert get("mean") == pytest.approx((L / ul).mean(), rel=1e-14)
    assert get("mean_volume") == pytest.approx(L.sum() / ul.sum(), rel=1e-14)


# ---------------------------------------------------------------- invariants

def test_invariants_on_random_ragged_batch(oracle_mod):
    rng = np.random.default_rng(5)
    durs = [0, 1, 2, 3]
    z, labels, tl, ul, blank = _random_case(rng, 4, 9, 5, 6, durs, sigma=0.1, ragged=True)
    tl = np.maximum(tl, 3)
    r = oracle_mod.tdt_loss(z, labels, tl, ul, durs, blank, 0.1, "none", want_lattice=True)
    lse, lpb, lpl, lpd = oracle_mod.node_tables(z, labels, tl, ul, len(durs), blank)
    V = z.shape[-1] - len(durs)
    np.testing.assert_allclose(r.ll_alpha, r.ll_beta, rtol=1e-13)
    g = r.grad
    # token and duration gradient rows each sum to zero
    assert np.abs(g[..., :V].sum(-1)).max() < 1e-12
    assert np.abs(g[..., V:].sum(-1)).max() < 1e-12
    assert g.min() >= -1 - 1e-12 and g.max() <= 1 + 1e-12
    for b in range(4):
        Tb, Ub = int(tl[b]), int(ul[b])
        occ = np.exp(r.alpha[b, :Tb, : Ub + 1] + r.beta[b, :Tb, : Ub + 1] - r.ll_alpha[b])
        sm = np.exp(z[b, :Tb, : Ub + 1, :V] - lse[b, :Tb, : Ub + 1, None])
        smd = np.exp(lpd[b, :Tb, : Ub + 1])
        # label posterior mass: every label is emitted exactly once
        for u in range(Ub):
            y = labels[b, u]
            gl = sm[:, u, y] * occ[:, u] - g[b, :Tb, u, y]
            assert gl.sum() == pytest.approx(1.0, abs=1e-12)
        # durations along any path add up to T_b
        gd = smd * occ[..., None] - g[b, :Tb, : Ub + 1, V:]
        assert (gd * np.array(durs)).sum() == pytest.approx(Tb, rel=1e-12)
        # blank posterior mass: arcs leaving row U_b are blanks, one path ends there
        gb = sm[:, Ub, blank] * occ[:, Ub] - g[b, :Tb, Ub, blank]
        assert gb.sum() >= 1.0 - 1e-12
        # start node is on every path
        assert occ[0, 0] == pytest.approx(1.0, abs=1e-12)


def test_loss_is_invariant_to_per_node_logit_shifts(oracle_mod):
    rng = np.random.default_rng(3)
    durs = [0, 1, 2]
    z, labels, tl, ul, blank = _random_case(rng, 2, 6, 3, 5, durs, sigma=0.3)
    V = 5
    base = oracle_mod.tdt_loss(z, labels, tl, ul, durs, blank, 0.3, "none", want_grad=False).loss
    z2 = z.copy()
    z2[0, 2, 1, :V] += 50.0
    z2[1, 4, 3, V:] -= 30.0
    z2[1, 0, 0, :V] += 7.0
    shifted = oracle_mod.tdt_loss(z2, labels, tl, ul, durs, blank, 0.3, "none",
                                  want_grad=False).loss
    np.testing.assert_allclose(shifted, base, rtol=1e-12)


def test_node_tables_match_scipy_log_softmax(oracle_mod):
    z, labels, tl, ul, w = _np_inputs("tiny")
    lse, lpb, lpl, lpd = oracle_mod.node_tables(z, labels, tl, ul, w.D, w.blank)
    zd = z.astype(np.float64)
    tok = log_softmax(zd[..., : w.V], axis=-1)
    np.testing.assert_allclose(lpb, tok[..., w.blank], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lpd, log_softmax(zd[..., w.V:], axis=-1), rtol=0, atol=1e-13)
    for b in range(w.B):
        for u in range(w.U):
            np.testing.assert_allclose(lpl[b, :, u], tok[b, :, u, labels[b, u]], atol=1e-13)
    assert np.isnan(lpl[:, :, w.U]).all()


# ---------------------------------------------------------------- degenerate cases

def test_no_path_gives_infinite_loss_and_zero_grad(oracle_mod):
    """durations [0, 2]: only even frames are reachable, so an odd T_b has no
    path; the reading is L_b = +inf with a zero gradient."""
    rng = np.random.default_rng(9)
    z, labels, tl, ul, blank = _random_case(rng, 2, 5, 2, 4, [0, 2])
    tl = np.array([5, 4])
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [0, 2], blank, 0.0, "none")
    assert r.utt_loss[0] == np.inf and np.isfinite(r.utt_loss[1])
    assert not r.grad[0].any()
    assert np.abs(r.grad[1]).sum() > 0


def test_unusable_utterances_give_nan(oracle_mod):
    rng = np.random.default_rng(10)
    z, labels, tl, ul, blank = _random_case(rng, 4, 5, 2, 4, [0, 1])
    labels[1, 0] = blank          # blank used as a label
    tl[2] = 6                     # longer than the tensor
    labels[3, 1] = 4              # out of the token range
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [0, 1], blank, 0.0, "none")
    assert np.isfinite(r.utt_loss[0])
    assert np.isnan(r.utt_loss[1:]).all()
    assert not r.grad[1:].any()


def test_empty_label_sequence(oracle_mod):
    """U_b = 0: the path is blanks only; with durations [1] the loss is
    T_b * (-log p_blank) summed, the plain product of per-frame blank probs."""
    rng = np.random.default_rng(12)
    z, labels, tl, ul, blank = _random_case(rng, 1, 6, 2, 4, [1])
    ul = np.array([0])
    r = oracle_mod.tdt_loss(z, labels, tl, ul, [1], blank, 0.0, "none")
    tok = log_softmax(z[0, :, 0, :4], axis=-1)
    assert r.utt_loss[0] == pytest.approx(-tok[:, blank].sum(), rel=1e-13)


def test_tiny_golden_file(oracle_mod):
    """Regression guard: tests/golden/tiny_oracle.json (written by
    tests/golden/make_golden.py, which calls only the oracle)."""
    import json
    import os

    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")))
    z, labels, tl, ul, w = _np_inputs("tiny")
    assert float(z.astype(np.float64).sum()) == pytest.approx(gold["logits_sum"], rel=1e-12)
    assert labels.tolist() == gold["labels"]
    r = oracle_mod.tdt_loss(z, labels, tl, ul, w.durations, w.blank, w.sigma, w.reduction)
    np.testing.assert_allclose(r.utt_loss, gold["utt_loss"], rtol=1e-13)
    assert float(np.abs(r.grad).sum()) == pytest.approx(gold["grad_abs_sum"], rel=1e-12)
