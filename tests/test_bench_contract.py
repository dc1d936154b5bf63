"""The benchmark's JSON contract, on the CPU.

`bench.py --impl reference` times the float64 oracle on the host cores and
prints one JSON line with the contract's keys; the GPU arm needs a CUDA
device and must fail (non-zero exit) rather than fall back to anything.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_the_contract_line():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_without_a_gpu():
    r = _run(["--workload", "tiny", "--steps", "2", "--warmup", "3", "--no-cpu-baseline"],
             timeout=120)
    assert r.returncode != 0
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def _bench_module():
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_counts_lattice_rows_read_and_every_row_written():
    """The roofline's numerator: every logit of a lattice row (t < T_b,
    u <= U_b) read once, every gradient element written once.  Checked
    against an explicit enumeration of the rows on a ragged bf16 view, and
    the parakeet figure from its sizes alone."""
    from transducer_loss_asr_gb300.workloads import WORKLOADS, scaled

    bench = _bench_module()
    w = scaled(WORKLOADS["parakeet_bf16_ragged"], name="bytes", B=3, T=7, U=4, V=20, blank=19,
               base_vd=30)
    tl = torch.tensor([7, 3, 5])
    ul = torch.tensor([4, 0, 2])
    read_b, write_b, valid, rows = bench.algorithmic_bytes(
        {"workload": w, "logit_lens": tl, "label_lens": ul})
    lattice_rows = sum(1 for b in range(3) for t in range(7) for u in range(5)
                       if t < int(tl[b]) and u <= int(ul[b]))
    assert valid == lattice_rows == 7 * 5 + 3 * 1 + 5 * 3
    assert rows == 3 * 7 * 5
    assert read_b == lattice_rows * w.VD * 2 and write_b == rows * w.VD * 2
    # parakeet fp32 [4, 200, 41, 8198], full lengths: 2 x 1,075,577,600 bytes
    p = WORKLOADS["parakeet"]
    read_b, write_b, _, _ = bench.algorithmic_bytes(
        {"workload": p, "logit_lens": torch.full((4,), 200), "label_lens": torch.full((4,), 40)})
    assert read_b == write_b == 1_075_577_600
    assert read_b + write_b == 2_151_155_200
