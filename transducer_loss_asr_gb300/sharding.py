"""Data-parallel TDT loss: the batch split by utterance across ranks.

Every utterance's lattice is independent, so ranks need no exchange of
tensors: each rank runs the loss on its own utterances and only two scalars
per rank are summed -- the utterance count and the label count, which the
batch-level reductions divide by -- plus, for reporting, the reduced loss
itself.  The gradient needs no extra pass: the split API's backward call
takes the rank's share of the global reduction as its upstream gradient.

For a reduction r over the global batch, the rank's local loss with the same
reduction times ``w`` is its share of the global loss, and ``w`` times its
local gradient is the gradient of the global loss w.r.t. its logits:
    sum          w = 1
    mean_batch   w = B_local / B_global          (c_b = 1 / B_global)
    mean         w = B_local / B_global          (c_b = 1 / (B_global U_b))
    mean_volume  w = sumU_local / sumU_global    (c_b = 1 / sumU_global)
    none         no combination: each rank keeps its utterances' losses.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_bounds(B: int, rank: int, world: int):
    """Contiguous utterance range [b0, b1) of ``rank``; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    return B * rank // world, B * (rank + 1) // world


def global_counts(label_lens: torch.Tensor, group=None) -> torch.Tensor:
    """[B_global, sumU_global] (float64, on label_lens' device) by one all-reduce;
    [B_local, sumU_local] when no process group is initialised."""
    counts = torch.stack([
        torch.tensor(float(label_lens.numel()), dtype=torch.float64, device=label_lens.device),
        label_lens.to(torch.float64).sum()])
    local = counts.clone()
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return torch.stack([local, counts])


def shard_weight(reduction: str, counts: torch.Tensor) -> torch.Tensor:
    """w (float32, one element) from ``global_counts``' [[B_l, U_l], [B_g, U_g]]."""
    (b_l, u_l), (b_g, u_g) = counts[0], counts[1]
    if reduction == "sum":
        w = torch.ones_like(b_l)
    elif reduction in ("mean", "mean_batch"):
        w = b_l / b_g
    elif reduction == "mean_volume":
        w = u_l / u_g
    else:
        raise ValueError("no weight for reduction %r" % reduction)
    return w.to(torch.float32).reshape(1)


def sharded_tdt_loss(logits, labels, logit_lens, label_lens, durations, blank, sigma=0.0,
                     reduction="mean_volume", group=None, fwd=None, bwd=None):
    """This rank's call of a loss over a batch sharded by utterance.

    Arguments are the rank's own utterances, as for the binding.  Returns
    (loss, grad): for reductions other than "none", the global reduced loss
    (the same on every rank) and the gradient of that loss w.r.t. this rank's
    logits; for "none", this rank's per-utterance losses and their gradient.
    ``fwd``/``bwd`` default to the library's split entry points
    (binding.tdt_loss_fwd / tdt_loss_bwd) and take the same arguments.
    """
    if fwd is None or bwd is None:
        from . import binding

        fwd = fwd or binding.tdt_loss_fwd
        bwd = bwd or binding.tdt_loss_bwd
    loss, ws = fwd(logits, labels, logit_lens, label_lens, durations, blank, sigma, reduction)
    if reduction == "none":
        grad = bwd(logits, labels, logit_lens, label_lens, durations, blank, ws, None, sigma,
                   reduction)
        return loss, grad
    w = shard_weight(reduction, global_counts(label_lens, group))
    grad = bwd(logits, labels, logit_lens, label_lens, durations, blank, ws, w, sigma, reduction)
    share = loss.reshape(1).to(torch.float64) * w.to(torch.float64)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(share, op=dist.ReduceOp.SUM, group=group)
    return share.to(torch.float32).reshape(()), grad
