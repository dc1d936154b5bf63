"""PyTorch autograd and torch.compile support for the TDT loss.

The loss is registered as two custom ops over the split C ABI
(``tdt_loss_fwd`` / ``tdt_loss_bwd`` in include/tdt_loss.h):

* ``tdt_gb300::tdt_loss_forward`` -> (loss, workspace): node tables, alpha,
  beta and the arc fractions; the workspace (uint8) carries them to the
  backward op.
* ``tdt_gb300::tdt_loss_backward`` -> grad: the gradient pass only, scaled by
  the upstream gradient of the loss, so an arbitrary ``grad_output`` costs no
  extra pass over the gradient.

Both have fake implementations (shapes only), so the ops trace under
torch.compile(fullgraph=True) and pass torch.library.opcheck.  The pages'
layer gained the same properties in review: backward support, then fake
implementations, opcheck and compiled-vs-eager tests ("Add TDT loss kernel",
transformers PR #46048, thread on the kernel mapping).  The ops have CUDA
kernels only: called with CPU tensors they raise.
"""
from __future__ import annotations

from typing import List, Tuple

import torch
from torch import Tensor

REDUCTIONS = ("none", "sum", "mean", "mean_batch", "mean_volume")


def _align(v):
    return (v + 255) // 256 * 256


def workspace_nbytes(B, T, U1, n_dur):
    """Bytes of the split API's workspace for logits [B, T, U1, V+D].

    The same value as the C ABI's tdt_loss_workspace_size, written with
    integer arithmetic only so that it also holds for symbolic sizes under
    torch.compile: per anti-diagonal slot a node arc record of 2 * D arc
    probabilities, alpha and beta (8 bytes each: int32 exponent, float32
    mantissa) and a record of 2 + D arc fractions (float32); per node two
    log-sum-exps; per utterance likelihood, scale, flag and the lattice
    launch's start counter; every region 256-byte aligned.
    """
    ndiag = B * (T + U1 - 1) * U1
    nodes = B * T * U1
    rec_len = 2 * n_dur
    regions = (ndiag * 8 * rec_len, ndiag * 8, ndiag * 8, nodes * 4, nodes * 4,
               ndiag * 4 * (2 + n_dur), B * 8, B * 4, B * 4, B * 4)
    off = 0
    for r in regions:
        off = _align(off + r)
    return torch.sym_max(off, 256)


@torch.library.custom_op("tdt_gb300::tdt_loss_forward", mutates_args=(), device_types="cuda")
def tdt_loss_forward(logits: Tensor, labels: Tensor, logit_lengths: Tensor,
                     label_lengths: Tensor, durations: List[int], blank: int, sigma: float,
                     reduction: str) -> Tuple[Tensor, Tensor]:
    from . import binding

    B, T, U1, _ = logits.shape
    loss = torch.empty((B,) if reduction == "none" else (), dtype=torch.float32,
                       device=logits.device)
    # zero-filled: the kernels leave slots of nodes outside a lattice
    # unwritten, and an op's outputs must be a function of its inputs
    # (torch.compile and opcheck compare them)
    ws = torch.zeros(int(workspace_nbytes(B, T, U1, len(durations))), dtype=torch.uint8,
                     device=logits.device)
    loss, ws = binding.tdt_loss_fwd(logits, labels, logit_lengths, label_lengths, durations,
                                    blank, sigma, reduction, loss_out=loss, workspace=ws)
    return loss, ws


@tdt_loss_forward.register_fake
def _tdt_loss_forward_fake(logits, labels, logit_lengths, label_lengths, durations, blank, sigma,
                           reduction):
    B, T, U1, _ = logits.shape
    loss = logits.new_empty((B,) if reduction == "none" else (), dtype=torch.float32)
    ws = logits.new_empty((workspace_nbytes(B, T, U1, len(durations)),), dtype=torch.uint8)
    return loss, ws


@torch.library.custom_op("tdt_gb300::tdt_loss_backward", mutates_args=(), device_types="cuda")
def tdt_loss_backward(grad_loss: Tensor, logits: Tensor, labels: Tensor, logit_lengths: Tensor,
                      label_lengths: Tensor, workspace: Tensor, durations: List[int], blank: int,
                      sigma: float, reduction: str) -> Tensor:
    from . import binding

    g = grad_loss.to(torch.float32).contiguous()
    return binding.tdt_loss_bwd(logits, labels, logit_lengths, label_lengths, durations, blank,
                                workspace, grad_loss=g, sigma=sigma, reduction=reduction)


@tdt_loss_backward.register_fake
def _tdt_loss_backward_fake(grad_loss, logits, labels, logit_lengths, label_lengths, workspace,
                            durations, blank, sigma, reduction):
    return torch.empty(logits.shape, dtype=logits.dtype, device=logits.device)


def _setup_context(ctx, inputs, output):
    logits, labels, logit_lengths, label_lengths, durations, blank, sigma, reduction = inputs
    _, ws = output
    ctx.save_for_backward(logits, labels, logit_lengths, label_lengths, ws)
    ctx.args = (list(durations), blank, sigma, reduction)


def _backward(ctx, grad_loss, grad_ws):
    logits, labels, logit_lengths, label_lengths, ws = ctx.saved_tensors
    durations, blank, sigma, reduction = ctx.args
    grad = tdt_loss_backward(grad_loss, logits, labels, logit_lengths, label_lengths, ws,
                             durations, blank, sigma, reduction)
    return grad, None, None, None, None, None, None, None


tdt_loss_forward.register_autograd(_backward, setup_context=_setup_context)


def tdt_loss(logits: Tensor, labels: Tensor, logit_lengths: Tensor, label_lengths: Tensor,
             durations, blank: int, sigma: float = 0.0, reduction: str = "mean_volume") -> Tensor:
    """TDT loss of ``logits`` [B, T, U+1, V+D] (CUDA; float32/float16/bfloat16,
    may be a slice ``base[..., :V+D]``), differentiable w.r.t. ``logits``.

    labels: int64 [B, U] (padding -100); logit_lengths, label_lengths: int64
    [B]; durations: list of D distinct ints; blank in [0, V); sigma: logit
    under-normalisation; reduction: none | sum | mean | mean_batch |
    mean_volume.  Returns float32 [B] for "none", else a 0-dim tensor.
    """
    if reduction not in REDUCTIONS:
        raise ValueError("reduction must be one of %s" % (REDUCTIONS,))
    loss, _ = tdt_loss_forward(logits, labels, logit_lengths, label_lengths,
                               [int(d) for d in durations], int(blank), float(sigma), reduction)
    return loss


class TDTLoss(torch.nn.Module):
    """Stateless module form of :func:`tdt_loss` (same arguments)."""

    def forward(self, logits, labels, logit_lengths, label_lengths, durations, blank,
                sigma=0.0, reduction="mean_volume"):
        return tdt_loss(logits, labels, logit_lengths, label_lengths, durations, blank, sigma,
                        reduction)
