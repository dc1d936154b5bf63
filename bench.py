#!/usr/bin/env python
"""Benchmark of the TDT loss forward+backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the C ABI (node tables, alpha, beta, reduction,
gradient) over one batch of the workload, inputs already in HBM.  L2 is
flushed (a 2x-L2 buffer is written) between timed steps, outside the events.
Prints one JSON line (rank 0).  ``value`` is achieved HBM throughput over the
algorithmic bytes of the step (valid-node logits read once + every gradient
element written once); ``ms_per_step`` the time of one step.  The steps are
timed twice: once as a user runs them (``value``, ``ms_per_step``), then
again with the library's per-kernel CUDA events for the per-kernel times, the
roofline of the gradient pass and the launch count (those events sit between
the kernels on their streams and lengthen the step by a few percent).

Under torchrun (N > 1) every rank runs its own replica of the workload (the
loss shards by utterance; there is no exchange on the path): weak scaling,
value = bytes of all ranks / max-over-ranks time.

``--impl reference`` times the CPU oracle (float64 C, OpenMP) on a bounded
sample of the same workload on the host cores; the other ranks exit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from transducer_loss_asr_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = ("TDT loss fwd+bwd ms and achieved HBM GB/s (% of roofline) at "
          "B4·T200·U40·V8193")
ELT = {"f32": 4, "f16": 2, "bf16": 2}
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the gradient kernel from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum), valid only while
# its sources hash to this sha256 (kernel_sha).
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch =
    # one utterance [1,200,41,8198] fp32 (the per-launch work of the
    # four-chunk B=4 bench): read 269417216 + written 213922816 bytes (the
    # rest of the writes retire from L2 after the kernel)
    ("grad", "parakeet"): {
        "bytes": 269417216 + 213922816,
        "sha256": "4d9371a502c0320e440b1c01a7654a673a86fe2e70cd9f88fd307f38b5a530e4",
    },
}


def algorithmic_bytes(inp):
    """Valid-node logits read once + every gradient element written once."""
    w = inp["workload"]
    tl = inp["logit_lens"].cpu().numpy()
    ul = inp["label_lens"].cpu().numpy()
    elt = ELT[w.dtype]
    valid_rows = int(np.sum(np.minimum(tl, w.T) * (np.minimum(ul, w.U) + 1)))
    all_rows = w.B * w.T * (w.U + 1)
    return valid_rows * w.VD * elt, all_rows * w.VD * elt, valid_rows, all_rows


def nominal_hbm_gbs(dev):
    """HBM bandwidth from the device's memory clock and bus width (double
    data rate), for context beside the measured copy peak; None if the
    attributes cannot be read."""
    prop = torch.cuda.get_device_properties(dev)
    clk, bus = getattr(prop, "memory_clock_rate", 0), getattr(prop, "memory_bus_width", 0)
    if not clk or not bus:
        try:  # the CUDA runtime the library already loaded
            import ctypes

            rt = None
            for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
                try:
                    rt = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            if rt is None:
                return None
            vals = []
            for attr in (36, 37):  # cudaDevAttrMemoryClockRate (kHz), ...GlobalMemoryBusWidth (bits)
                v = ctypes.c_int(0)
                if rt.cudaDeviceGetAttribute(ctypes.byref(v), attr, dev.index or 0) != 0:
                    return None
                vals.append(v.value)
            clk, bus = vals
        except Exception:
            return None
    if not clk or not bus:
        return None
    return clk * 1e3 * 2 * bus / 8 / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_SOURCES = {"grad": ("tdt_grad.cu", "tdt_rowio.cuh", "tdt_async.cuh", "tdt_common.cuh")}


def kernel_sha(kernel):
    """sha256 over the sources a kernel is compiled from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "transducer_loss_asr_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def oracle_sample(inp, max_utts=1, frames=None):
    """The oracle on the first utterance(s) of the workload, float32 up-cast;
    ``frames`` keeps only that many leading frames (a smaller bounded sample)."""
    import oracle

    w = inp["workload"]
    b = min(max_utts, w.B)
    T = w.T if frames is None else max(1, min(frames, w.T))
    z = inp["logits"][:b, :T].float().cpu().numpy()
    labels = inp["labels"][:b].cpu().numpy()
    tl = np.minimum(inp["logit_lens"][:b].cpu().numpy(), T)
    ul = inp["label_lens"][:b].cpu().numpy()
    elt = ELT[w.dtype]
    valid = int(np.sum(tl * (ul + 1)))
    sample_bytes = valid * w.VD * elt + b * T * (w.U + 1) * w.VD * elt
    oracle.build()

    def run():
        if w.loss == "rnnt":
            oracle.rnnt_loss(z, labels, tl, ul, inp["blank"], inp["sigma"], inp["reduction"])
        else:
            oracle.tdt_loss(z, labels, tl, ul, inp["durations"], inp["blank"], inp["sigma"],
                            inp["reduction"])

    return run, sample_bytes, "%d of %d utterances, %d of %d frames (%d lattice rows of %d)" % (
        b, w.B, T, w.T, valid, w.B * w.T * (w.U + 1))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = make_inputs(w, device="cpu")
    run, sample_bytes, desc = oracle_sample(inp)
    t0 = time.perf_counter()
    run()
    t1 = time.perf_counter() - t0
    budget = 120.0  # seconds for warmup + timed steps
    if (args.steps + args.warmup) * t1 > budget:
        frames = int(w.T * budget / ((args.steps + args.warmup) * t1))
        run, sample_bytes, desc = oracle_sample(inp, frames=frames)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = sample_bytes / dt / 1e9
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, "oracle on host cores"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_decode(args, w, inp, dev, world, rank, dist):
    """Time greedy TDT decoding of the workload's logits (one call = the
    whole batch).  Each step of an utterance is a dependent row read plus a
    block-wide argmax, so the call is latency-bound: reported in ms and in
    decoded tokens per second."""
    from transducer_loss_asr_gb300 import binding

    def step():
        return binding.tdt_greedy_decode(inp["logits"], inp["logit_lens"], inp["durations"],
                                         inp["blank"], args.max_symbols)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        n = step()[0]
    torch.cuda.synchronize()
    tokens = int(n.sum().item())
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    if rank == 0:
        print(json.dumps({
            "metric": "greedy TDT decode of precomputed joint outputs, ms per batch",
            "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(config_dict(w, "flushed between timed steps (2x L2 write)", world),
                           max_symbols=args.max_symbols),
            "tokens_per_batch": tokens, "tokens_per_s": world * tokens / (ms / 1e3),
            "roofline": {"bound": "latency", "note": "one dependent row read and block argmax "
                         "per step; T_b + U + 1 steps at most per utterance"},
            "gpu_launches": args.steps}))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def config_dict(w, l2, world=1):
    """The workload per rank; with N ranks each runs its own replica (the loss
    shards by utterance), so the global batch is N x B."""
    return {"workload": "%s: B%d T%d U%d V%d D%d %s [%d,%d,%d,%d]%s, sigma %g, %s" % (
        w.name, w.B, w.T, w.U, w.V, w.D, w.dtype, w.B, w.T, w.U + 1, w.VD,
        " view of width %d" % w.base_vd if w.base_vd else "", w.sigma, w.reduction),
        "lengths": "full" if w.T_range is None else "T_b in %s, U_b in %s" % (w.T_range,
                                                                             w.U_range),
        "l2": l2, "global_batch": w.B * world, "loss": w.loss,
        "parallelism": "one GPU" if world == 1 else
                       "dp%d: one replica per GPU, no data-path collective" % world}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="parakeet", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (smaller profiling cases; not a bench line)")
    ap.add_argument("--frames", type=int, default=None,
                    help="override T (smaller profiling cases; not a bench line)")
    ap.add_argument("--op", default="loss", choices=["loss", "decode"],
                    help="loss: TDT loss fwd+bwd (the benchmark); decode: greedy TDT decoding "
                         "of the workload's logits (a separate measurement)")
    ap.add_argument("--max-symbols", type=int, default=10)
    ap.add_argument("--lattice-bands", type=int, default=0,
                    help="force K row bands per utterance in the lattice passes (0: automatic)")
    ap.add_argument("--lattice-exchange", type=int, default=0,
                    help="how lattice bands exchange boundary rows: 0 automatic, "
                         "1 thread-block cluster, 2 global memory (tuning)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.batch is not None or args.frames is not None:
        from transducer_loss_asr_gb300.workloads import scaled

        ch = {}
        if args.batch is not None:
            ch["B"] = args.batch
        if args.frames is not None:
            ch["T"] = args.frames
            if w.T_range is not None:
                ch["T_range"] = (min(w.T_range[0], args.frames), args.frames)
        w = scaled(w, name="%s_%s" % (w.name, "_".join("%s%d" % (k, v) for k, v in ch.items()
                                                         if k != "T_range")), **ch)
    if args.impl == "reference":
        return run_reference(args, w)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    from transducer_loss_asr_gb300 import binding

    binding.tdt_loss_set_lattice_bands(args.lattice_bands)
    binding.tdt_loss_set_lattice_exchange(args.lattice_exchange)
    inp = make_inputs(w, device=dev, seed=w.seed + rank)
    if args.op == "decode":
        return run_decode(args, w, inp, dev, world, rank, dist)
    logits = inp["logits"]
    read_b, write_b, valid_rows, all_rows = algorithmic_bytes(inp)
    step_bytes = read_b + write_b
    loss = torch.empty(w.B if w.reduction == "none" else 1, dtype=torch.float32, device=dev)
    grad = torch.empty(logits.shape, dtype=logits.dtype, device=dev)

    def call(z, labels, tl, ul):
        if w.loss == "rnnt":
            binding.tdt_rnnt_loss_fwd_bwd(z, labels, tl, ul, inp["blank"], inp["sigma"],
                                          inp["reduction"], loss_out=loss, grad_out=grad)
        else:
            binding.tdt_loss_fwd_bwd(z, labels, tl, ul, inp["durations"], inp["blank"],
                                     inp["sigma"], inp["reduction"], loss_out=loss,
                                     grad_out=grad)

    def step():
        call(logits, inp["labels"], inp["logit_lens"], inp["label_lens"])

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def timed_steps(kernel_events):
        """K steps, L2 flushed before each (outside the events), CUDA events
        around each step on the launching stream; returns the summed ms.
        With kernel_events the library also records events around each of
        its kernels (on the stream each runs on) -- they sit between the
        kernels on the streams and lengthen the step, so the headline step
        time comes from a run without them."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        binding.tdt_loss_timing_read(reset=True)
        binding.tdt_loss_timing_enable(kernel_events)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xff)
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        binding.tdt_loss_timing_enable(False)
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends))

    # headline: the steps as a user runs them (no per-kernel events)
    sampler = ClockSampler(local) if local == 0 else None
    if sampler:
        sampler.start()
    total_ms = timed_steps(False)
    if sampler:
        sampler.stop()
    # per-kernel breakdown, roofline and launch count: the same steps again
    # with the library's per-kernel events
    kernel_step_ms = timed_steps(True) / args.steps
    kt = binding.tdt_loss_timing_read(reset=True)
    t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = world * step_bytes * args.steps / (total_ms / 1e3) / 1e9

    # end to end through host buffers: the step's inputs host -> device from
    # pinned memory, the call, the step's result (the loss) device -> host;
    # the gradient stays on the device, where the backward pass of the joint
    # network consumes it.  Two device input buffers: step i + 1's copy (on a
    # copy stream) runs while step i computes, as a data loader would; every
    # step's copy and loss read lie inside the timed region.
    e2e_steps = args.e2e_steps or min(args.steps, 20)
    base = logits._base if logits._base is not None else logits
    base_h = torch.empty(base.shape, dtype=base.dtype, pin_memory=True)
    base_h.copy_(base)
    labels_h = inp["labels"].cpu().pin_memory()
    tl_h = inp["logit_lens"].cpu().pin_memory()
    ul_h = inp["label_lens"].cpu().pin_memory()
    bufs = []
    for _ in range(2):
        base_d = torch.empty_like(base)
        bufs.append((base_d, base_d[..., : w.VD] if base is not logits else base_d,
                     torch.empty_like(inp["labels"]), torch.empty_like(inp["logit_lens"]),
                     torch.empty_like(inp["label_lens"])))
    loss_h = torch.empty(loss.shape, dtype=loss.dtype, pin_memory=True)
    h2d = (base_h.numel() * base_h.element_size() + labels_h.numel() * 8 + tl_h.numel() * 8
           + ul_h.numel() * 8)
    d2h = loss_h.numel() * 4
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]   # buffer k holds its step's inputs
    free = [torch.cuda.Event(), torch.cuda.Event()]    # the call that read buffer k is done

    def copy_in(k, first_use):
        base_d, _, labels_d, tl_d, ul_d = bufs[k]
        with torch.cuda.stream(copier):
            if not first_use:
                copier.wait_event(free[k])
            base_d.copy_(base_h, non_blocking=True)
            labels_d.copy_(labels_h, non_blocking=True)
            tl_d.copy_(tl_h, non_blocking=True)
            ul_d.copy_(ul_h, non_blocking=True)
            ready[k].record(copier)

    def e2e_run(n):
        copier.wait_stream(compute)
        copy_in(0, True)
        for i in range(n):
            k = i & 1
            if i + 1 < n:
                copy_in(k ^ 1, i == 0)
            compute.wait_event(ready[k])
            _, view_d, labels_d, tl_d, ul_d = bufs[k]
            call(view_d, labels_d, tl_d, ul_d)
            free[k].record(compute)
            loss_h.copy_(loss, non_blocking=True)
        compute.wait_stream(copier)

    e2e_run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record()
    e2e_run(e2e_steps)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = torch.tensor([e0.elapsed_time(e1) / e2e_steps], dtype=torch.float64, device=dev)
    if dist is not None:
        dist.all_reduce(e2e_ms, op=dist.ReduceOp.MAX)
    e2e_value = world * step_bytes / (float(e2e_ms.item()) / 1e3) / 1e9
    assert torch.equal(loss_h, loss.cpu())

    # Roofline of the gradient pass (K4), the largest HBM-bound share of the
    # step; the lattice passes are latency-bound, run on SMs of their own and
    # overlap K1/K4 (their share is reported beside it).  The K4 launches of a
    # step (one per chunk) run on two streams and overlap one another's
    # tails, so K4's time per step is its busy window (first launch start to
    # last launch end, CUDA events on the launching streams) and the bytes are
    # the step's algorithmic bytes; per launch, both are divided by the K4
    # launches per step.
    per_kernel = {k: {"ms_per_launch": (ms / n if n else 0.0), "launches": n,
                      "busy_ms_per_step": span / args.steps}
                  for k, (ms, n, span) in kt.items()}
    peak, peak_kind = measured_peaks()
    roofline = None
    ms_g, n_g, span_g = kt.get("grad", (0.0, 0, 0.0))
    k4_bytes = read_b + write_b
    if n_g and span_g > 0:
        per_step = n_g / args.steps
        bytes_launch = k4_bytes / per_step
        achieved = k4_bytes * args.steps / (span_g / 1e3) / 1e9
        tr = NCU_TRAFFIC.get(("grad", w.name))
        traffic = tr["bytes"] if tr and tr["sha256"] == kernel_sha("grad") else None
        roofline = {"bound": "hbm", "kernel": "grad", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                    "algorithmic_bytes_per_launch": bytes_launch,
                    "launches_per_step": per_step,
                    "time": "K4 busy window per step / launches per step",
                    "bytes_per_step": k4_bytes,
                    "peak_source": peak_kind + " hbm_gbs (copy)"}
    ms_t, n_t, span_t = kt.get("node_tables", (0.0, 0, 0.0))
    if n_t and span_t > 0:
        per_kernel["node_tables"]["achieved_gbs"] = read_b * args.steps / (span_t / 1e3) / 1e9
    if roofline:
        per_kernel["grad"]["achieved_gbs"] = roofline["achieved"]
    nominal = nominal_hbm_gbs(dev)
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    if roofline:
        # the node-table pass (K1): the second, dependency-forced read of the
        # lattice rows, over its busy window per step; and the whole step
        # over the metric's bytes, against the same measured copy peak
        if "achieved_gbs" in per_kernel.get("node_tables", {}):
            k1 = per_kernel["node_tables"]["achieved_gbs"]
            roofline["node_tables"] = {"achieved": k1, "frac": k1 / peak, "unit": "GB/s",
                                       "bytes_per_step": read_b,
                                       "time": "K1 busy window per step"}
        roofline["step"] = {"achieved": step_gbs, "frac": step_gbs / peak, "unit": "GB/s",
                            "bytes_per_step": step_bytes, "time": "ms_per_step",
                            "frac_of_nominal_hbm": step_gbs / nominal if nominal else None}
    # the lattice passes are latency-bound: T_b + U_b dependent anti-diagonal
    # steps per utterance (alpha and beta run side by side); report the time
    # per step of the longest utterance of a launch
    if "lattice" in per_kernel and per_kernel["lattice"]["launches"]:
        steps = int((inp["logit_lens"].clamp(max=w.T) + inp["label_lens"].clamp(max=w.U)).max())
        per_kernel["lattice"]["bound"] = "latency"
        per_kernel["lattice"]["diagonal_steps"] = steps
        per_kernel["lattice"]["us_per_diagonal_step"] = (
            per_kernel["lattice"]["ms_per_launch"] * 1e3 / max(steps, 1))
    step_frac = (step_bytes / (ms_per_step / 1e3) / 1e9) / peak

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        run, sample_bytes, desc = oracle_sample(inp)
        run()  # warm: build + page in
        reps, t0 = 0, time.perf_counter()
        while reps < 3 or time.perf_counter() - t0 < 10.0:
            run()
            reps += 1
            if time.perf_counter() - t0 > 30.0:
                break
        dt = (time.perf_counter() - t0) / reps
        cpu = {"value": sample_bytes / dt / 1e9, "unit": "GB/s", "cores": host_cores(),
               "kind": "oracle", "sample": desc + ", %d runs, %.2f s each" % (reps, dt)}

    if rank == 0:
        clocks = sampler.summary() if sampler else None
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": config_dict(w, "flushed between timed steps (2x L2 write)", world),
            "frac_of_hbm_roofline": step_frac,
            "frac_of_measured_copy_peak": step_frac,
            "frac_of_nominal_hbm": step_gbs / nominal if nominal else None,
            "measured_copy_peak_gbs": peak,
            "nominal_hbm_gbs": nominal,
            "algorithmic_bytes_per_step": step_bytes,
            "roofline": roofline,
            "kernels": per_kernel,
            "kernel_timing": ("a second timed run of the same steps with per-kernel CUDA events "
                              "(its step: %.4f ms); value and ms_per_step come from the run "
                              "without them" % kernel_step_ms),
            "gpu_launches": int(sum(v[1] for v in kt.values())),
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": float(e2e_ms.item()),
                    "steps": e2e_steps},
            "clocks": clocks,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
