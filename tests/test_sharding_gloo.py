"""The data-parallel path on CPU: two gloo ranks, each with its shard of a
ragged batch, run ``sharded_tdt_loss`` with the float64 oracle standing in
for the library's forward/backward calls.  The global loss and every rank's
gradient must equal the oracle on the whole batch -- this checks the shard
bounds, the count all-reduce and the per-reduction weights of the host
logic (the GPU path differs only in the fwd/bwd callables)."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DURS = [0, 1, 2, 3]
BLANK = 7
SIGMA = 0.03


def _batch():
    g = np.random.default_rng(20261205)
    B, T, U, VD = 5, 7, 4, 8 + len(DURS)
    logits = g.normal(0.0, 1.5, size=(B, T, U + 1, VD)).astype(np.float32)
    tl = np.array([7, 5, 6, 3, 7], dtype=np.int64)
    ul = np.array([4, 2, 3, 1, 0], dtype=np.int64)
    labels = np.full((B, U), -100, dtype=np.int64)
    for b in range(B):
        labels[b, : ul[b]] = g.integers(0, BLANK, size=ul[b])
    return logits, labels, tl, ul


def _oracle_fwd_bwd():
    import oracle

    state = {}

    def fwd(logits, labels, tl, ul, durations, blank, sigma, reduction):
        r = oracle.tdt_loss(logits.numpy(), labels.numpy(), tl.numpy(), ul.numpy(), durations,
                            blank, sigma, reduction, want_grad=True)
        state["grad"] = r.grad
        return torch.from_numpy(np.asarray(r.loss, dtype=np.float64)), "ws"

    def bwd(logits, labels, tl, ul, durations, blank, ws, grad_loss, sigma, reduction):
        assert ws == "ws"
        g = torch.from_numpy(state["grad"])
        if grad_loss is not None:
            g = g * grad_loss.to(torch.float64).reshape(-1)[0]
        return g

    return fwd, bwd


def _worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    from transducer_loss_asr_gb300.sharding import shard_bounds, sharded_tdt_loss

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        logits, labels, tl, ul = _batch()
        b0, b1 = shard_bounds(logits.shape[0], rank, world)
        fwd, bwd = _oracle_fwd_bwd()
        res = {}
        for red in ("sum", "mean", "mean_batch", "mean_volume", "none"):
            loss, grad = sharded_tdt_loss(
                torch.from_numpy(logits[b0:b1]), torch.from_numpy(labels[b0:b1]),
                torch.from_numpy(tl[b0:b1]), torch.from_numpy(ul[b0:b1]), DURS, BLANK, SIGMA,
                red, fwd=fwd, bwd=bwd)
            res[red] = (loss.numpy().astype(np.float64), grad.numpy())
        np.save(os.path.join(out_dir, "rank%d.npy" % rank),
                np.array([b0, b1, res], dtype=object), allow_pickle=True)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_batch():
    from transducer_loss_asr_gb300.sharding import shard_bounds

    for B in range(0, 13):
        for world in range(1, 6):
            spans = [shard_bounds(B, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_whole_batch(oracle_mod):
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_worker, args=(world, _free_port(), d), nprocs=world, join=True,
                           start_method="spawn")
        parts = [np.load(os.path.join(d, "rank%d.npy" % r), allow_pickle=True)
                 for r in range(world)]
    logits, labels, tl, ul = _batch()
    for red in ("sum", "mean", "mean_batch", "mean_volume", "none"):
        ref = oracle_mod.tdt_loss(logits, labels, tl, ul, DURS, BLANK, SIGMA, red)
        if red == "none":
            got = np.concatenate([p[2][red][0] for p in parts])
            np.testing.assert_allclose(got, ref.loss, rtol=1e-12)
        else:
            for p in parts:  # every rank holds the global loss
                np.testing.assert_allclose(p[2][red][0], ref.loss[0], rtol=1e-6)
        for p in parts:
            b0, b1 = int(p[0]), int(p[1])
            np.testing.assert_allclose(p[2][red][1], ref.grad[b0:b1], rtol=1e-6, atol=1e-7)
