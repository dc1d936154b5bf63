"""Pins of the plain RNN-T oracle (oracle/rnnt_oracle.c): brute-force path
enumeration, the closed form for uniform logits, central finite
differences, invariants, and the one case where the TDT oracle computes the
same thing (no labels, durations [1])."""
import math

import numpy as np
import pytest

from lattice_pins import log_softmax


def _inputs(seed, B, T, U, V, blank, ragged=False, std=1.5):
    g = np.random.default_rng(seed)
    z = g.normal(0.0, std, size=(B, T, U + 1, V))
    tl = g.integers(1, T + 1, size=B) if ragged else np.full(B, T)
    ul = g.integers(0, U + 1, size=B) if ragged else np.full(B, U)
    labels = np.full((B, U), -100, dtype=np.int64)
    for b in range(B):
        y = g.integers(0, V - 1, size=ul[b])
        labels[b, : ul[b]] = y + (y >= blank)
    return z, labels, tl.astype(np.int64), ul.astype(np.int64)


def _brute_force(z, labels, Tb, Ub, blank, sigma):
    """log of the summed weight of every RNN-T alignment, path by path."""
    lp = log_softmax(z, axis=-1)
    total = []

    def walk(t, u, acc):
        if t == Tb - 1 and u == Ub:
            total.append(acc + lp[t, u, blank] - sigma)  # the final blank
        if t + 1 < Tb:
            walk(t + 1, u, acc + lp[t, u, blank] - sigma)
        if u < Ub:
            walk(t, u + 1, acc + lp[t, u, labels[u]] - sigma)

    walk(0, 0, 0.0)
    m = max(total)
    return m + math.log(sum(math.exp(x - m) for x in total)), len(total)


@pytest.mark.parametrize("seed,T,U,sigma", [(1, 5, 3, 0.0), (2, 7, 4, 0.13), (3, 4, 0, 0.0),
                                            (4, 1, 3, 0.05), (5, 6, 6, -0.2)])
def test_brute_force(oracle_mod, seed, T, U, sigma):
    z, labels, tl, ul = _inputs(seed, 1, T, U, 6, blank=2)
    ref, npaths = _brute_force(z[0], labels[0], T, U, 2, sigma)
    assert npaths == math.comb(T - 1 + U, U)
    r = oracle_mod.rnnt_loss(z, labels, tl, ul, blank=2, sigma=sigma, reduction="none")
    assert abs(-r.loss[0] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_brute_force_ragged_batch(oracle_mod):
    z, labels, tl, ul = _inputs(11, 4, 6, 4, 5, blank=0, ragged=True)
    r = oracle_mod.rnnt_loss(z, labels, tl, ul, blank=0, sigma=0.07, reduction="none")
    for b in range(4):
        ref, _ = _brute_force(z[b], labels[b], tl[b], ul[b], 0, 0.07)
        assert abs(-r.loss[b] - ref) <= 1e-12 * max(1.0, abs(ref))


@pytest.mark.parametrize("T,U,V,sigma", [(40, 30, 7, 0.0), (300, 200, 33, 0.02),
                                         (1000, 1, 5, 0.0)])
def test_closed_form_uniform_logits(oracle_mod, T, U, V, sigma):
    # every arc has log-prob -log V - sigma; a path has T blanks and U labels;
    # there are C(T+U-1, U) paths
    z = np.zeros((1, T, U + 1, V))
    labels = np.ones((1, U), dtype=np.int64)
    r = oracle_mod.rnnt_loss(z, labels, [T], [U], blank=0, sigma=sigma, reduction="none")
    want = (T + U) * (math.log(V) + sigma) - (math.lgamma(T + U) - math.lgamma(U + 1)
                                              - math.lgamma(T))
    assert abs(r.loss[0] - want) <= 1e-10 * want


@pytest.mark.parametrize("reduction", ["none", "sum", "mean", "mean_batch", "mean_volume"])
def test_finite_differences(oracle_mod, reduction):
    z, labels, tl, ul = _inputs(7, 2, 4, 2, 5, blank=4, ragged=True)
    ul = np.maximum(ul, 1)
    r = oracle_mod.rnnt_loss(z, labels, tl, ul, blank=4, sigma=0.1, reduction=reduction)

    def f(zz):
        return oracle_mod.rnnt_loss(zz, labels, tl, ul, blank=4, sigma=0.1, reduction=reduction,
                                    want_grad=False).loss.sum()

    h = 1e-5
    num = np.zeros_like(z)
    it = np.nditer(z, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        zp = z.copy(); zp[i] += h
        zm = z.copy(); zm[i] -= h
        num[i] = (f(zp) - f(zm)) / (2 * h)
    np.testing.assert_allclose(r.grad, num, atol=2e-7, rtol=1e-6)


def test_invariants(oracle_mod):
    z, labels, tl, ul = _inputs(9, 3, 9, 5, 8, blank=7, ragged=True)
    r = oracle_mod.rnnt_loss(z, labels, tl, ul, blank=7, sigma=0.0, reduction="sum",
                             want_lattice=True)
    np.testing.assert_allclose(r.ll_alpha, r.ll_beta, rtol=1e-12)
    np.testing.assert_allclose(r.grad.sum(axis=-1), 0.0, atol=1e-12)
    for b in range(3):
        occ = np.exp(r.alpha[b, : tl[b], : ul[b] + 1] + r.beta[b, : tl[b], : ul[b] + 1]
                     - r.ll_alpha[b])
        # every path visits T_b + U_b nodes; (0,0) and (T_b-1, U_b) on all of them
        assert abs(occ.sum() - (tl[b] + ul[b])) <= 1e-9 * (tl[b] + ul[b])
        assert abs(occ[0, 0] - 1.0) <= 1e-12 and abs(occ[-1, -1] - 1.0) <= 1e-12
        assert not r.grad[b, tl[b]:].any() and not r.grad[b, :, ul[b] + 1:].any()


def test_unusable_and_shift_invariance(oracle_mod):
    z, labels, tl, ul = _inputs(13, 2, 5, 3, 6, blank=5)
    bad = labels.copy(); bad[1, 0] = 5  # a label equal to blank
    r = oracle_mod.rnnt_loss(z, bad, tl, ul, blank=5, reduction="none")
    assert np.isfinite(r.loss[0]) and np.isnan(r.loss[1]) and not r.grad[1].any()
    z2 = z.copy(); z2[0, 2, 1] += 40.0  # one node's logits shifted: same loss
    a = oracle_mod.rnnt_loss(z, labels, tl, ul, blank=5, reduction="none", want_grad=False)
    c = oracle_mod.rnnt_loss(z2, labels, tl, ul, blank=5, reduction="none", want_grad=False)
    np.testing.assert_allclose(a.loss, c.loss, rtol=1e-12)


def test_matches_tdt_oracle_without_labels(oracle_mod):
    # with U = 0 and durations [1], every TDT path is T blanks with duration
    # log-prob 0: the TDT loss is the RNN-T loss of the token logits
    g = np.random.default_rng(21)
    z = g.normal(size=(2, 9, 1, 6))
    zt = np.concatenate([z, g.normal(size=(2, 9, 1, 1))], axis=-1)
    labels = np.zeros((2, 0), dtype=np.int64)
    r = oracle_mod.rnnt_loss(z, labels, [9, 7], [0, 0], blank=3, sigma=0.3, reduction="none")
    t = oracle_mod.tdt_loss(zt, labels, [9, 7], [0, 0], [1], 3, 0.3, "none")
    np.testing.assert_allclose(r.loss, t.loss, rtol=1e-12)
    np.testing.assert_allclose(r.grad, t.grad[..., :6], atol=1e-13)
