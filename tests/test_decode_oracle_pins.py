"""Pins of the greedy TDT decoding oracle (oracle/decode.py): decoding
logits in which a chosen path was planted must return that path; the
structural rules (timestamps, the per-frame symbol guard, stopping) hold on
random logits."""
import numpy as np
import pytest

from oracle.decode import tdt_greedy_decode

DURS = [0, 1, 2, 3, 4]


def _plant(path, T, U, V, D, seed, blank):
    """Random logits in [-1, 1) with, at each visited node, the planted token
    and duration index raised to +5."""
    g = np.random.default_rng(seed)
    z = g.uniform(-1, 1, size=(1, T, U + 1, V + D))
    for (t, u, k, di) in path:
        z[0, t, u, k] = 5.0
        z[0, t, u, V + di] = 5.0
    return z


def test_planted_path():
    # frames: t=0 emit 3 (d 0), emit 5 (d 2) -> t=2 blank (d 1) -> t=3 emit 1 (d 3) -> t=6
    # blank (d 0 -> moves 1) -> t=7 >= T = 7: stop
    V, D, blank = 8, 5, 7
    path = [(0, 0, 3, 0), (0, 1, 5, 2), (2, 2, blank, 1), (3, 2, 1, 3), (6, 3, blank, 0)]
    z = _plant(path, T=7, U=4, V=V, D=D, seed=1, blank=blank)
    n, tok, fr, du = tdt_greedy_decode(z, [7], DURS, blank, max_symbols=10)
    assert n[0] == 3
    assert tok[0, :3].tolist() == [3, 5, 1]
    assert fr[0, :3].tolist() == [0, 0, 3]
    assert du[0, :3].tolist() == [0, 2, 3]
    assert tok[0, 3:].tolist() == [-1, -1]


def test_symbol_guard_forces_a_frame_step():
    # the planted path emits with duration 0 forever at frame 0; with
    # max_symbols = 2 the second emission moves to frame 1
    V, D, blank = 6, 5, 5
    path = [(0, 0, 2, 0), (0, 1, 3, 0), (1, 2, 4, 0), (1, 3, 1, 0), (2, 4, blank, 2)]
    z = _plant(path, T=4, U=5, V=V, D=D, seed=2, blank=blank)
    n, tok, fr, du = tdt_greedy_decode(z, [4], DURS, blank, max_symbols=2)
    assert tok[0, :4].tolist() == [2, 3, 4, 1]
    assert fr[0, :4].tolist() == [0, 0, 1, 1]
    assert n[0] == 4


def test_stops_when_rows_run_out():
    V, D, blank = 5, 5, 4
    path = [(0, 0, 1, 0), (0, 1, 2, 0), (0, 2, 3, 1)]  # U = 2: three emissions, then no row
    z = _plant(path, T=9, U=2, V=V, D=D, seed=3, blank=blank)
    n, tok, fr, _ = tdt_greedy_decode(z, [9], DURS, blank, max_symbols=10)
    assert n[0] == 3 and tok[0].tolist() == [1, 2, 3] and fr[0].tolist() == [0, 0, 0]


def test_ties_take_the_first_index():
    z = np.zeros((1, 3, 2, 4 + 2))       # every logit equal: token 0, duration index 0
    n, tok, fr, du = tdt_greedy_decode(z, [3], [2, 1], blank=3, max_symbols=5)
    # token 0 (not blank) with duration 2 at t = 0 -> u = 1 at t = 2 -> token 0 again -> stop
    assert n[0] == 2 and tok[0].tolist() == [0, 0] and fr[0].tolist() == [0, 2]
    assert du[0].tolist() == [2, 2]


@pytest.mark.parametrize("seed", range(5))
def test_structure_on_random_logits(seed):
    g = np.random.default_rng(seed)
    B, T, U, V = 6, 30, 12, 10
    durs = [0, 1, 2, 4]
    z = g.normal(size=(B, T, U + 1, V + len(durs)))
    z[..., 0] += 0.5  # make blank (index 0) frequent
    tl = g.integers(1, T + 1, size=B)
    n, tok, fr, du = tdt_greedy_decode(z, tl, durs, blank=0, max_symbols=3)
    for b in range(B):
        k = n[b]
        assert 0 <= k <= U + 1
        assert (tok[b, :k] != 0).all() and (tok[b, k:] == -1).all()
        f = fr[b, :k]
        assert (np.diff(f) >= 0).all() and (f < tl[b]).all()
        assert all(np.sum(f == x) <= 3 for x in set(f.tolist()))
        assert set(du[b, :k].tolist()) <= set(durs)
