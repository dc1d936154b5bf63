"""The schedule of the global-exchange lattice bands, replayed on the CPU.

When a lattice is too tall for one CTA, its rows are split into bands that
pass their boundary row to the neighbouring band through global memory
(csrc/tdt_lattice.cu, kXGlobal).  This test restates that schedule in
plain Python, step by step as each band's CTA runs it, and interleaves the
bands at random:

- a band keeps the values of its rows (and of the neighbour's boundary row)
  for the last RA diagonals in a ring of RA slots (slot q mod RA);
- the neighbour's value of diagonal q is copied into the ring with the arc
  records of diagonal q, P diagonals ahead of use -- possibly before the
  neighbour has written it, in which case the copy holds the "unwritten"
  marker;
- during the step of diagonal q the band checks that copy and, only if it
  still holds the marker, polls global memory until the neighbour's value
  is there; the value is used from the next step on;
- CTAs take their role from a start-order ticket (ticket j of an utterance:
  alpha band j / 2, or beta band K - 1 - j / 2), and at most R of them are
  resident at once, admitted in ticket order: a band only ever waits on a
  band with a smaller ticket, so the schedule cannot deadlock;
- a band wholly above the utterance's label count leaves at once.

Alpha and beta (probabilities, float64) must equal the oracle's log-domain
lattice, for random lengths, duration sets, band sizes, P and R.  The arc
weights come from the oracle's node tables, so nothing here restates the
loss's arithmetic beyond the arc-weight product of the lattice recursion.
"""
import math
import random

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

MARK = None  # the unwritten marker in "global memory" and in a ring slot


def pow2_at_least(v):
    r = 1
    while r < v:
        r <<= 1
    return r


def alpha_band(k, K, Rc, Tb, Ub, durs, WB, WL, G_alpha, RA, P):
    """One alpha band's CTA: yields 'wait' while polling, 'step' per diagonal."""
    u_lo = k * Rc
    if u_lo > Ub:
        return
    nsteps = Tb + Ub
    lower = k > 0
    uh = u_lo - 1
    ring = [[0.0] * RA for _ in range(Rc + 2)]

    def halo_node(q):
        return lower and 0 <= q - uh < Tb and uh <= Ub

    def fetch(q):  # the boundary value's copy, with the records of diagonal q
        if halo_node(q):
            ring[0][q % RA] = G_alpha.get((q, uh), MARK)

    for q in range(P):
        fetch(q)
    for s in range(nsteps):
        fetch(s + P)
        vals = []
        for row in range(1, Rc + 1):
            u = u_lo + row - 1
            t = s - u
            node = u <= Ub and 0 <= t < Tb
            v = 0.0
            if node and s == 0:
                v = 1.0
            elif node:
                for i, d in enumerate(durs):
                    tb = t - d
                    if d > 0 and tb >= 0:
                        v += ring[row][(s - d) % RA] * WB[tb, u, i]
                    if u >= 1 and tb >= 0:
                        src = ring[row - 1][(s - d - 1) % RA]
                        assert src is not MARK, "read a boundary value before its check"
                        v += src * WL[tb, u - 1, i]
            vals.append((row, u, node, v))
        for row, u, node, v in vals:
            ring[row][s % RA] = v
            if node:
                G_alpha[(s, u)] = v
        # the check of the copy of diagonal s, one step before its use
        if lower:
            if not halo_node(s):
                ring[0][s % RA] = 0.0
            elif ring[0][s % RA] is MARK:
                while (s, uh) not in G_alpha:
                    yield "wait"
                ring[0][s % RA] = G_alpha[(s, uh)]
        yield "step"


def beta_band(k, K, Rc, Tb, Ub, durs, WB, WL, G_beta, RA, P):
    u_lo = k * Rc
    if u_lo > Ub:
        return
    nsteps = Tb + Ub
    last = nsteps - 1
    upper = k + 1 < K
    uh = u_lo + Rc
    ring = [[0.0] * RA for _ in range(Rc + 2)]
    for row in range(1, Rc + 1):
        if u_lo + row - 1 == Ub:
            ring[row][nsteps % RA] = 1.0  # the end state (T_b, U_b)

    def halo_node(q):
        return upper and 0 <= q - uh < Tb and uh <= Ub

    def fetch(q):
        if halo_node(q):
            ring[Rc + 1][q % RA] = G_beta.get((q, uh), MARK)

    for i in range(P):
        fetch(last - i)
    for i in range(nsteps):
        q = last - i
        fetch(q - P)
        vals = []
        for row in range(1, Rc + 1):
            u = u_lo + row - 1
            t = q - u
            node = u <= Ub and 0 <= t < Tb
            v = 0.0
            if node:
                for j, d in enumerate(durs):
                    if d > 0:
                        v += ring[row][(q + d) % RA] * WB[t, u, j]
                    if q < Tb + u - d:  # a label arc lands before T_b
                        dst = ring[row + 1][(q + d + 1) % RA]
                        assert dst is not MARK, "read a boundary value before its check"
                        v += dst * WL[t, u, j]
            vals.append((row, u, node, v))
        for row, u, node, v in vals:
            ring[row][q % RA] = v
            if node:
                G_beta[(q, u)] = v
        if upper:
            if not halo_node(q):
                ring[Rc + 1][q % RA] = 0.0
            elif ring[Rc + 1][q % RA] is MARK:
                while (q, uh) not in G_beta:
                    yield "wait"
                ring[Rc + 1][q % RA] = G_beta[(q, uh)]
        yield "step"


def run_schedule(Tb, Ub, durs, WB, WL, Rc, P, resident, rng):
    U1 = Ub + 1
    K = (U1 + Rc - 1) // Rc
    RA = pow2_at_least(max(durs) + 10)
    assert RA > P + max(durs) + 1
    G_alpha, G_beta = {}, {}
    # ticket j -> role: alpha band j / 2 (even j), beta band K - 1 - j / 2 (odd j)
    roles = []
    for j in range(2 * K):
        band = j >> 1
        if j & 1:
            roles.append(beta_band(K - 1 - band, K, Rc, Tb, Ub, durs, WB, WL, G_beta, RA, P))
        else:
            roles.append(alpha_band(band, K, Rc, Tb, Ub, durs, WB, WL, G_alpha, RA, P))
    pending = list(range(len(roles)))  # admitted in ticket order
    running = []
    idle = 0
    while pending or running:
        while pending and len(running) < resident:
            running.append(pending.pop(0))
        j = rng.choice(running)
        try:
            event = next(roles[j])
        except StopIteration:
            running.remove(j)
            idle = 0
            continue
        idle = idle + 1 if event == "wait" else 0
        assert idle < 100000, "no resident band can progress"
    return G_alpha, G_beta


@pytest.mark.parametrize("seed", range(40))
def test_global_band_schedule_matches_oracle_lattice(oracle_mod, seed):
    rng = random.Random(seed)
    nrng = np.random.default_rng(seed)
    T = rng.randint(1, 9)
    U = rng.randint(1, 14)
    V = 6
    nd = rng.randint(1, 4)
    durs = sorted(rng.sample(range(0, 7), nd))
    if max(durs) == 0:
        durs = [0, 1]
    Tb, Ub = rng.randint(1, T), rng.randint(0, U)
    logits = nrng.normal(0.0, 1.5, size=(1, T, U + 1, V + len(durs))).astype(np.float64)
    labels = nrng.integers(0, V - 1, size=(1, U)).astype(np.int64)  # blank = V - 1 unused
    tl = np.array([Tb], dtype=np.int64)
    ul = np.array([Ub], dtype=np.int64)
    sigma = 0.02
    ref = oracle_mod.tdt_loss(logits, labels, tl, ul, durs, V - 1, sigma, "none",
                              want_grad=False, want_lattice=True)
    _, lpb, lpl, lpd = oracle_mod.node_tables(logits, labels, tl, ul, len(durs), V - 1)
    with np.errstate(invalid="ignore"):
        WB = np.nan_to_num(np.exp(lpb[0][..., None] - sigma + lpd[0]), nan=0.0)
        WL = np.nan_to_num(np.exp(lpl[0][..., None] - sigma + lpd[0]), nan=0.0)
    WL[:, Ub:, :] = 0.0  # no label arc leaves row U_b (its target is not a node)
    Rc = rng.randint(1, 4)
    P = rng.choice([2, 4, 8])
    K = (Ub + 1 + Rc - 1) // Rc
    resident = rng.randint(1, 2 * K)
    G_alpha, G_beta = run_schedule(Tb, Ub, durs, WB, WL, Rc, P, resident, rng)
    for t in range(Tb):
        for u in range(Ub + 1):
            for got, want in ((G_alpha[(t + u, u)], ref.alpha[0, t, u]),
                              (G_beta[(t + u, u)], ref.beta[0, t, u])):
                if want == -math.inf:
                    assert got == 0.0
                else:
                    assert abs(math.log(got) - want) <= 1e-9 * max(1.0, abs(want)), (t, u)


def test_global_band_schedule_resident_limit_one():
    """With one resident CTA at a time the bands run strictly in ticket
    order, and every wait still ends: a band's producer always has a smaller
    ticket."""
    rng = random.Random(7)
    T, U, durs = 5, 9, [0, 1, 3]
    WB = np.full((T, U + 1, len(durs)), 0.3)
    WL = np.full((T, U + 1, len(durs)), 0.2)
    G_alpha, G_beta = run_schedule(T, U, durs, WB, WL, Rc=2, P=4, resident=1, rng=rng)
    assert len(G_alpha) == T * (U + 1) and len(G_beta) == T * (U + 1)
