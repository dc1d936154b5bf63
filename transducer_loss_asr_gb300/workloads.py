"""Seeded synthetic inputs for the TDT loss (no loss arithmetic lives here).

The only workload the pages measure is "loss fwd+bwd at Parakeet size: batch
4, 200 frames, 40 labels, vocab 8193" ("tdt-loss: add TDT loss kernel",
kernels-community PR #882, benchmark table), plus a fine-tune on LibriSpeech
that needs a dataset and trained weights.  Random joint-network outputs of the
same shapes stand in for both; the five named workloads below also cover the
features the pages list (bf16 input, a no-copy slice ``logits[..., :V+D]`` of
a wider tensor, ragged lengths with -100 label padding, sigma != 0, every
reduction, label sequences longer than 1024).

Recipe (all integers uniform and inclusive; "N(0, s)" has standard deviation s):
  logits  = randn(shape, generator seeded with ``seed``) * std in float32,
            then cast to the workload dtype (the cast tensor is the input);
            a ``base_vd`` wider than V+D makes the input the view
            ``base[..., :V+D]``
  labels  = uniform over the V-1 tokens other than blank (drawn in [0, V-2],
            values >= blank shifted up by one; blank = V-1 in every named
            workload, where this is uniform in [0, blank-1]), entries at
            u >= U_b set to -100
  T_b, U_b = full, or uniform in the stated ranges
Integers come from a CPU generator seeded with ``seed + 1`` so that they do
not depend on the device.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    U: int                      # maximum label count; lattice has U+1 rows
    V: int                      # token logits, blank inside
    blank: int
    durations: tuple
    dtype: str                  # "f32" | "f16" | "bf16"
    std: float
    sigma: float
    reduction: str
    T_range: tuple | None = None   # (lo, hi) inclusive, None = full
    U_range: tuple | None = None
    base_vd: int | None = None     # width of the wider tensor the input is sliced from
    seed: int = BASE_SEED
    loss: str = "tdt"              # "tdt" | "rnnt" (plain RNN-T: no duration head)
    notes: str = field(default="", compare=False)

    @property
    def D(self) -> int:
        return len(self.durations)

    @property
    def VD(self) -> int:
        return self.V + self.D

    @property
    def shape(self):
        return (self.B, self.T, self.U + 1, self.VD)


WORKLOADS = {
    "tiny": Workload(
        "tiny", B=2, T=12, U=4, V=9, blank=8, durations=(0, 1, 2, 3), dtype="f32", std=2.0,
        sigma=0.0, reduction="none", seed=BASE_SEED + 0,
        notes="B2 T12 U4 V9 D4 fp32 N(0,2); small enough for brute-force path enumeration"),
    "parakeet": Workload(
        "parakeet", B=4, T=200, U=40, V=8193, blank=8192, durations=(0, 1, 2, 3, 4), dtype="f32",
        std=1.0, sigma=0.0, reduction="mean_volume", seed=BASE_SEED + 1,
        notes="B4 T200 U40 V8193 D5 fp32 [4,200,41,8198], full lengths: the pages' benchmark size"),
    "parakeet_bf16_ragged": Workload(
        "parakeet_bf16_ragged", B=4, T=200, U=40, V=8193, blank=8192, durations=(0, 1, 2, 3, 4),
        dtype="bf16", std=1.0, sigma=0.05, reduction="mean_batch", T_range=(100, 200),
        U_range=(10, 40), base_vd=8205, seed=BASE_SEED + 2,
        notes="bf16 view [..., :8198] of [4,200,41,8205], ragged lengths, -100 padding"),
    "large_batch": Workload(
        "large_batch", B=16, T=750, U=120, V=1025, blank=1024, durations=(0, 1, 2, 3, 4),
        dtype="bf16", std=1.5, sigma=0.0, reduction="sum", T_range=(600, 750), U_range=(90, 120),
        seed=BASE_SEED + 3, notes="B16 T750 U120 V1025 bf16 N(0,1.5), ragged"),
    "long_labels": Workload(
        "long_labels", B=1, T=2000, U=1200, V=129, blank=128, durations=tuple(range(9)),
        dtype="f32", std=1.0, sigma=0.02, reduction="none", seed=BASE_SEED + 4,
        notes="B1 T2000 U1200 V129 D9 fp32: labels beyond 1024, long float64 lattice"),
    "parakeet_rnnt": Workload(
        "parakeet_rnnt", B=4, T=200, U=40, V=8193, blank=8192, durations=(), dtype="f32",
        std=1.0, sigma=0.0, reduction="mean_volume", seed=BASE_SEED + 5, loss="rnnt",
        notes="plain RNN-T loss (no duration head) at the pages' benchmark size [4,200,41,8193]"),
}

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (e.g. smaller T for CPU tests)."""
    return replace(w, **changes)


def make_inputs(w: Workload | str, device="cpu", seed: int | None = None):
    """Build the seeded inputs of a workload on ``device``.

    Returns a dict with logits (the input tensor, possibly a strided view),
    labels [B, U] int64, logit_lens [B] int64, label_lens [B] int64,
    durations (list of int), blank, sigma, reduction.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    seed = w.seed if seed is None else seed
    device = torch.device(device)
    vd = w.base_vd if w.base_vd is not None else w.VD
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    base = torch.randn((w.B, w.T, w.U + 1, vd), generator=gen, device=device,
                       dtype=torch.float32)
    if w.std != 1.0:
        base.mul_(w.std)
    base = base.to(TORCH_DTYPES[w.dtype])
    logits = base[..., : w.VD] if vd != w.VD else base

    ig = torch.Generator(device="cpu")
    ig.manual_seed(seed + 1)
    if w.T_range is None:
        logit_lens = torch.full((w.B,), w.T, dtype=torch.int64)
    else:
        logit_lens = torch.randint(w.T_range[0], w.T_range[1] + 1, (w.B,), generator=ig)
    if w.U_range is None:
        label_lens = torch.full((w.B,), w.U, dtype=torch.int64)
    else:
        label_lens = torch.randint(w.U_range[0], w.U_range[1] + 1, (w.B,), generator=ig)
    labels = torch.randint(0, w.V - 1, (w.B, max(w.U, 0)), generator=ig, dtype=torch.int64)
    labels = labels + (labels >= w.blank).to(torch.int64)
    if w.U > 0:
        pad = torch.arange(w.U)[None, :] >= label_lens[:, None]
        labels = labels.masked_fill(pad, -100)
    return dict(
        logits=logits,
        labels=labels.to(device),
        logit_lens=logit_lens.to(device),
        label_lens=label_lens.to(device),
        durations=list(w.durations),
        blank=w.blank,
        sigma=w.sigma,
        reduction=w.reduction,
        workload=w,
    )
