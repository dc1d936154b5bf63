"""Greedy TDT decoding over precomputed joint outputs -- TEST INFRASTRUCTURE.

Only the tests use this module; the product never imports it.

Source: "Add TDT loss kernel" (transformers PR #46048), commit list: greedy
TDT decoding with per-token timestamps and token durations, and a guard on
the number of symbols emitted per frame ("max_symbols_per_step").  The
pages print no decoding loop; with the joint output z[t, u, :] given for
every frame t and every decoder state u (u tokens emitted so far), the
plainest reading of greedy TDT decoding is this walk:

    t, u, n_here = 0, 0, 0
    while t < T_b:
        k = first argmax of z[t, u, 0:V]          (token)
        d = durations[first argmax of z[t, u, V:V+D]]
        if k != blank:
            emit (k, frame t, duration d); u += 1; n_here += 1
            if u > U: stop                        (no joint output beyond row U)
        if d == 0 and (k == blank or n_here >= max_symbols): d = 1
        if d > 0: t += d; n_here = 0

A blank always moves on (a blank of duration 0 moves one frame), and at
most max_symbols tokens are emitted at one frame.  Written as plain Python
over numpy rows (a few hundred steps per utterance).
"""
from __future__ import annotations

import numpy as np


def tdt_greedy_decode(logits: np.ndarray, logit_lens, durations, blank: int, max_symbols: int):
    """logits [B, T, U+1, V+D] (float32 or float64, any strides); returns
    (n [B], tokens [B, U+1], frames [B, U+1], token_durations [B, U+1]) as
    int32 arrays, -1 past n[b]."""
    B, T, U1, VD = logits.shape
    D = len(durations)
    V = VD - D
    n = np.zeros(B, dtype=np.int32)
    tokens = np.full((B, U1), -1, dtype=np.int32)
    frames = np.full((B, U1), -1, dtype=np.int32)
    tdur = np.full((B, U1), -1, dtype=np.int32)
    for b in range(B):
        Tb = int(logit_lens[b])
        t = u = here = 0
        while t < Tb:
            row = logits[b, t, u]
            k = int(np.argmax(row[:V]))           # numpy: first maximum
            d = int(durations[int(np.argmax(row[V:]))])
            if k != blank:
                j = n[b]
                tokens[b, j], frames[b, j], tdur[b, j] = k, t, d
                n[b] += 1
                u += 1
                here += 1
                if u >= U1:
                    break
            if d == 0 and (k == blank or here >= max_symbols):
                d = 1
            if d > 0:
                t += d
                here = 0
    return n, tokens, frames, tdur
