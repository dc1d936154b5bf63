"""Independent evaluations of the TDT path sum, used to pin the oracle.

Nothing here shares code with ``oracle/`` or with the CUDA library.  Two
formulations that do not use the alpha/beta recursion:

* ``enumerate_paths``: the literal definition -- walk every alignment path
  from (0, 0) to the end of the lattice and add up exp(path weight).
* ``path_sum_linear``: the lattice as a weighted DAG with transfer matrix M
  (M[src, dst] = summed probability of the arcs src -> dst); the sum over all
  paths from s to e is [(I - M)^{-1}]_{s, e} (a library linear solve), which
  gives the total, the forward sums F = e_start (I - M)^{-1} and the backward
  sums G = (I - M)^{-1} e_end at every node.

Arc rules (the plain reading of the TDT lattice): blank (t,u)->(t+d,u) for
d > 0; label (t,u)->(t+d,u+1) for every d incl. 0, landing before frame T_b;
the path ends with a blank that lands exactly on T_b from row U_b.  Arc
weight: token log-prob - sigma + duration log-prob.
"""
from __future__ import annotations

import numpy as np
from scipy.special import log_softmax, logsumexp


def node_log_probs(z: np.ndarray, V: int, blank: int, labels, T: int, U: int):
    """Log-softmax tables of one utterance from its logits z[t, u, :] (float64)."""
    z = np.asarray(z, dtype=np.float64)
    tok = log_softmax(z[:T, : U + 1, :V], axis=-1)
    dur = log_softmax(z[:T, : U + 1, V:], axis=-1)
    lpb = tok[:, :, blank]
    lpl = np.full((T, U + 1), np.nan)
    for u in range(U):
        lpl[:, u] = tok[:, u, labels[u]]
    return lpb, lpl, dur


def arcs_from(t, u, T, U, durations):
    """Outgoing arcs of node (t, u): (kind, i, dst) with dst None for the end."""
    out = []
    for i, d in enumerate(durations):
        if d > 0:
            if t + d < T:
                out.append(("blank", i, (t + d, u)))
            elif t + d == T and u == U:
                out.append(("blank", i, None))
        if u < U and t + d < T:
            out.append(("label", i, (t + d, u + 1)))
    return out


def enumerate_paths(lpb, lpl, lpd, T, U, durations, sigma=0.0, count_only=False):
    """Sum over every alignment path, by explicit enumeration.

    Returns (log path sum, number of paths).  Iterative DFS; each complete
    path contributes exp(sum of its arc weights).
    """
    arcs = {}
    for t in range(T):
        for u in range(U + 1):
            lst = []
            for kind, i, dst in arcs_from(t, u, T, U, durations):
                tok = lpb[t, u] if kind == "blank" else lpl[t, u]
                lst.append((tok + lpd[t, u, i] - sigma, dst))
            arcs[(t, u)] = lst
    scores = []
    stack = [((0, 0), 0.0)]
    n_paths = 0
    while stack:
        node, acc = stack.pop()
        for w, dst in arcs[node]:
            if dst is None:
                n_paths += 1
                if not count_only:
                    scores.append(acc + w)
            else:
                stack.append((dst, acc + w))
    if count_only:
        return None, n_paths
    if not scores:
        return -np.inf, 0
    return float(logsumexp(np.array(scores))), n_paths


def path_sum_linear(lpb, lpl, lpd, T, U, durations, sigma=0.0):
    """Path sums through the transfer matrix of the lattice DAG.

    Returns (log Z, log F[t,u], log G[t,u]) where F is the summed weight of
    all partial paths (0,0) -> (t,u) and G of all suffixes (t,u) -> end.
    """
    idx = {}
    for t in range(T):
        for u in range(U + 1):
            idx[(t, u)] = len(idx)
    end = len(idx)
    n = end + 1
    M = np.zeros((n, n))
    for (t, u), s in idx.items():
        for kind, i, dst in arcs_from(t, u, T, U, durations):
            tok = lpb[t, u] if kind == "blank" else lpl[t, u]
            p = np.exp(tok + lpd[t, u, i] - sigma)
            M[s, end if dst is None else idx[dst]] += p
    A = np.eye(n) - M
    start = idx[(0, 0)]
    e_start = np.zeros(n); e_start[start] = 1.0
    e_end = np.zeros(n); e_end[end] = 1.0
    F = np.linalg.solve(A.T, e_start)   # row vector e_start (I-M)^{-1}
    G = np.linalg.solve(A, e_end)       # column (I-M)^{-1} e_end
    Z = F[end]
    with np.errstate(divide="ignore"):
        logF = np.log(np.array([[max(F[idx[(t, u)]], 0.0) for u in range(U + 1)]
                                for t in range(T)]))
        logG = np.log(np.array([[max(G[idx[(t, u)]], 0.0) for u in range(U + 1)]
                                for t in range(T)]))
        return float(np.log(Z)) if Z > 0 else -np.inf, logF, logG
