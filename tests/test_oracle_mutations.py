"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one (a dropped term, a wrong sign or index, a swapped operand).

Each mutant is compiled from a text substitution of ``oracle/tdt_oracle.c``
into a temporary directory; the oracle's own source is never modified.
"""
import math
import os
import subprocess

import numpy as np
import pytest
from scipy.special import gammaln

import oracle
from lattice_pins import enumerate_paths, node_log_probs, path_sum_linear

SRC = os.path.join(os.path.dirname(oracle.__file__), "tdt_oracle.c")

MUTANTS = {
    "sigma_dropped_on_label_arcs": (
        "return tb->lp_label[n] + tb->lp_dur[n * p->D + i] - p->sigma;",
        "return tb->lp_label[n] + tb->lp_dur[n * p->D + i];"),
    "sigma_added_not_subtracted": (
        "return tb->lp_blank[n] + tb->lp_dur[n * p->D + i] - p->sigma;",
        "return tb->lp_blank[n] + tb->lp_dur[n * p->D + i] + p->sigma;"),
    "no_same_frame_label_arcs": (
        "if (u >= 1) { /* label arc",
        "if (u >= 1 && d > 0) { /* label arc"),
    "duration_index_reversed": (
        "return tb->lp_blank[n] + tb->lp_dur[n * p->D + i] - p->sigma;",
        "return tb->lp_blank[n] + tb->lp_dur[n * p->D + (p->D - 1 - i)] - p->sigma;"),
    "final_blank_may_overshoot": (
        "else if (t + d == Tb && u == Ub) terms[k++] = w_blank(p, tb, n, i);",
        "else if (u == Ub) terms[k++] = w_blank(p, tb, n, i);"),
    "beta_label_arc_wrong_row": (
        "terms[k++] = beta[node_id(p, b, t + d, u + 1)] + w_label(p, tb, n, i);",
        "terms[k++] = beta[node_id(p, b, t + d, u)] + w_label(p, tb, n, i);"),
    "grad_blank_and_label_swapped": (
        "if (k == p->blank) v -= gb_sum;",
        "if (k == p->blank) v -= gl_sum;"),
    "grad_scale_dropped": (
        "g[k] = c * v;",
        "g[k] = v;"),
    "mean_not_divided_by_batch": (
        "case OR_RED_MEAN: cb[b] = 1.0 / ((double)p.B * (double)label_lens[b]); break;",
        "case OR_RED_MEAN: cb[b] = 1.0 / (double)label_lens[b]; break;"),
    "log_sum_exp_unshifted": (
        "for (int i = 0; i < n; ++i) s += exp(x[i] - m);",
        "for (int i = 0; i < n; ++i) s += exp(x[i]);"),
    "duration_grad_sign": (
        "g[p->V + i] = c * (smd * occ - gd[i]);",
        "g[p->V + i] = c * (gd[i] - smd * occ);"),
    "label_read_one_row_late": (
        "i64 y = p->labels[b * p->labels_stride + u];\n        tb->lp_label[n] = buf[y] - lse;",
        "i64 y = p->labels[b * p->labels_stride + (u + 1 < p->label_lens[b] ? u + 1 : u)];\n"
        "        tb->lp_label[n] = buf[y] - lse;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(old, new))
    lib = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(lib),
                    str(path), "-lm"], check=True)
    return oracle.load_library(str(lib))


def _pins_fail(lib) -> list:
    """Run a small battery of pins with ``lib``; return the names that fail."""
    failed = []
    rng = np.random.default_rng(42)
    durs = [0, 1, 2]
    B, T, U, V = 2, 5, 2, 4
    D = len(durs)
    z = rng.normal(0, 1.5, size=(B, T, U + 1, V + D))
    blank = V - 1
    labels = rng.integers(0, blank, size=(B, U)).astype(np.int64)
    tl = np.array([5, 4]); ul = np.array([2, 1])
    labels[1, 1:] = -100
    sigma = 0.2
    r = oracle.tdt_loss(z, labels, tl, ul, durs, blank, sigma, "none", want_lattice=True, lib=lib)
    # brute force and linear system
    for b in range(B):
        lpb, lpl, lpd = node_log_probs(z[b], V, blank, labels[b], int(tl[b]), int(ul[b]))
        ll, _ = enumerate_paths(lpb, lpl, lpd, int(tl[b]), int(ul[b]), durs, sigma)
        if not np.isclose(r.utt_loss[b], -ll, rtol=1e-12):
            failed.append("brute_force")
        lz, lF, lG = path_sum_linear(lpb, lpl, lpd, int(tl[b]), int(ul[b]), durs, sigma)
        a = r.alpha[b, : tl[b], : ul[b] + 1]
        bt = r.beta[b, : tl[b], : ul[b] + 1]
        if not (np.allclose(np.nan_to_num(a, neginf=-1e300), np.nan_to_num(lF, neginf=-1e300),
                            atol=1e-9)
                and np.allclose(np.nan_to_num(bt, neginf=-1e300),
                                np.nan_to_num(lG, neginf=-1e300), atol=1e-9)):
            failed.append("linear_system")
    if not np.allclose(r.ll_alpha, r.ll_beta, rtol=1e-12):
        failed.append("alpha_beta_agree")
    # finite differences for two reductions
    for red in ("none", "mean"):
        rr = oracle.tdt_loss(z, labels, tl, ul, durs, blank, sigma, red, lib=lib)
        flat = z.reshape(-1)
        fd = np.zeros_like(flat)
        for j in range(flat.size):
            old = flat[j]
            flat[j] = old + 1e-5
            lp = oracle.tdt_loss(z, labels, tl, ul, durs, blank, sigma, red, want_grad=False,
                                 lib=lib).loss.sum()
            flat[j] = old - 1e-5
            lm = oracle.tdt_loss(z, labels, tl, ul, durs, blank, sigma, red, want_grad=False,
                                 lib=lib).loss.sum()
            flat[j] = old
            fd[j] = (lp - lm) / 2e-5
        if not np.allclose(rr.grad.reshape(-1), fd, atol=1e-6):
            failed.append("finite_differences_" + red)
    # closed form, durations [1]
    T2, U2, V2 = 9, 4, 5
    zu = np.zeros((1, T2, U2 + 1, V2 + 1))
    r1 = oracle.tdt_loss(zu, np.zeros((1, U2), np.int64), np.array([T2]), np.array([U2]), [1],
                         V2 - 1, 0.1, "none", want_grad=False, lib=lib)
    expect = T2 * (math.log(V2) + 0.1) - (gammaln(T2) - gammaln(U2 + 1) - gammaln(T2 - U2))
    if not np.isclose(r1.utt_loss[0], expect, rtol=1e-12):
        failed.append("closed_form")
    return failed


def test_unmutated_oracle_passes_battery(oracle_mod):
    assert _pins_fail(None) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, oracle_mod, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    assert _pins_fail(lib), "planted mistake %r was not caught by any pin" % name
