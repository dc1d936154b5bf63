"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before touching any device (no GPU here:
only calls that fail validation are made)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from transducer_loss_asr_gb300 import build

    build.build()
    from transducer_loss_asr_gb300 import binding

    return binding


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(tdt_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = _declared_functions()
    for n in ("tdt_loss_fwd_bwd", "tdt_loss_fwd_bwd_ws", "tdt_loss_workspace_size",
              "tdt_loss_fwd", "tdt_loss_bwd", "tdt_status_string", "tdt_loss_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(so, n), n
        assert hasattr(lib, n), "binding lacks " + n


def test_version_and_status_strings(lib):
    assert lib.tdt_loss_version() == 1
    assert lib.tdt_status_string(0) == "ok"
    for code in range(-13, 0):
        assert lib.tdt_status_string(code) != "unknown status"
    assert lib.tdt_status_string(-99) == "unknown status"


def test_workspace_size(lib):
    s = lib.tdt_loss_workspace_size([4, 200, 41, 8198], 5)
    ndiag = 4 * (200 + 41 - 1) * 41
    nodes = 4 * 200 * 41
    assert s >= ndiag * 8 * (4 + 5) + nodes * 4 * (4 + 5)
    assert s % 256 == 0
    assert lib.tdt_loss_workspace_size([4, 200, 41, 8198], 0) == 0
    assert lib.tdt_loss_workspace_size([4, 0, 41, 8198], 5) == 0
    assert lib.tdt_loss_workspace_size([1, 60000, 6000, 10], 5) == 0   # T + U + 1 > 65536
    assert lib.tdt_loss_workspace_size([0, 5, 3, 10], 2) > 0           # empty batch is valid


FAKE = 0x10000  # never dereferenced: every call below fails host validation


def _call(lib, **over):
    so = lib.lib
    a = dict(logits=FAKE, sizes=[2, 5, 3, 10], strides=[150, 30, 10, 1], dtype=0, labels=FAKE,
             logit_lens=FAKE, label_lens=FAKE, durations=[0, 1, 2], blank=6, sigma=0.0,
             reduction=4, loss_out=FAKE, grad_out=FAKE)
    a.update(over)
    durs = a["durations"]
    n_dur = over.get("n_dur", len(durs))
    darr = (ctypes.c_int32 * max(1, len(durs)))(*durs) if durs is not None else None
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    sizes = None if a["sizes"] is None else (ctypes.c_int64 * 4)(*a["sizes"])
    strides = None if a["strides"] is None else (ctypes.c_int64 * 4)(*a["strides"])
    return so.tdt_loss_fwd_bwd(vp(a["logits"]), sizes, strides, a["dtype"], vp(a["labels"]),
                               vp(a["logit_lens"]), vp(a["label_lens"]), darr, n_dur,
                               a["blank"], a["sigma"], a["reduction"], vp(a["loss_out"]),
                               vp(a["grad_out"]), None)


@pytest.mark.parametrize("over,code", [
    (dict(sizes=None), -1),
    (dict(strides=None), -1),
    (dict(loss_out=None), -1),
    (dict(logits=None), -1),
    (dict(logit_lens=None), -1),
    (dict(labels=None), -1),
    (dict(dtype=3), -4),
    (dict(dtype=-1), -4),
    (dict(sizes=[2, 0, 3, 10]), -2),
    (dict(sizes=[2, 5, 0, 10]), -2),
    (dict(sizes=[-1, 5, 3, 10]), -2),
    (dict(sizes=[2, 5, 3, 3]), -2),             # V + D must exceed n_dur
    (dict(sizes=[1, 60000, 6000, 10]), -2),     # T + U + 1 > 65536
    (dict(sizes=[1 << 20, 64, 32, 10]), -2),    # B * T * (U+1) >= 2^31
    (dict(strides=[150, 30, 10, 2]), -3),
    (dict(strides=[150, -30, 10, 1]), -3),
    (dict(durations=[]), -5),
    (dict(durations=[0, 1, 1]), -5),            # duplicates
    (dict(durations=[0, -1]), -5),
    (dict(durations=[0, 256]), -5),
    (dict(durations=list(range(33))), -5),
    (dict(blank=7), -6),                         # V = 10 - 3 = 7
    (dict(blank=-1), -6),
    (dict(reduction=5), -7),
    (dict(sigma=float("nan")), -8),
    (dict(sigma=2000.0), -8),
    (dict(logits=FAKE + 2), -11),                # fp32 logits not 4-byte aligned
    (dict(grad_out=FAKE + 1, dtype=2), -11),
    (dict(grad_out=FAKE + 4), -13),              # overlaps the logits, not in place
    (dict(grad_out=FAKE, strides=[160, 32, 10, 1]), -13),  # in place over strided logits
])
def test_host_validation_rejects(lib, over, code):
    assert _call(lib, **over) == code


def test_labels_may_be_null_without_labels(lib):
    # U = 0: labels are not needed; with sizes otherwise invalid the call is
    # still rejected for the other reason, never for labels.
    assert _call(lib, labels=None, sizes=[2, 5, 1, 10], strides=[50, 10, 10, 1], dtype=7) == -4


def test_ws_variant_checks_workspace(lib):
    so = lib.lib
    sizes = (ctypes.c_int64 * 4)(2, 5, 3, 10)
    strides = (ctypes.c_int64 * 4)(150, 30, 10, 1)
    durs = (ctypes.c_int32 * 3)(0, 1, 2)
    need = lib.tdt_loss_workspace_size([2, 5, 3, 10], 3)
    f = ctypes.c_void_p(FAKE)
    args = [f, sizes, strides, 0, f, f, f, durs, 3, 6, 0.0, 4, f, f]
    assert so.tdt_loss_fwd_bwd_ws(*args, None, need, None) == -1
    assert so.tdt_loss_fwd_bwd_ws(*args, f, need - 1, None) == -9
    assert so.tdt_loss_fwd_bwd_ws(*args, ctypes.c_void_p(FAKE + 16), need, None) == -11


def test_binding_rejects_bad_tensors(lib):
    import torch

    z = torch.zeros(2, 5, 3, 10, dtype=torch.float64)
    with pytest.raises(TypeError):
        lib.tdt_loss_fwd_bwd(z, None, None, None, [0, 1], 0)
    with pytest.raises(ValueError):
        lib.tdt_loss_fwd_bwd(torch.zeros(5, 3, 10), None, None, None, [0, 1], 0)


def test_split_entry_points_validate(lib):
    so = lib.lib
    sizes = (ctypes.c_int64 * 4)(2, 5, 3, 10)
    strides = (ctypes.c_int64 * 4)(150, 30, 10, 1)
    durs = (ctypes.c_int32 * 3)(0, 1, 2)
    need = lib.tdt_loss_workspace_size([2, 5, 3, 10], 3)
    f = ctypes.c_void_p(FAKE)
    head = [f, sizes, strides, 0, f, f, f, durs, 3, 6, 0.0, 4]
    # forward: loss_out required, workspace checked
    assert so.tdt_loss_fwd(*head, None, f, need, None) == -1
    assert so.tdt_loss_fwd(*head, f, f, need - 1, None) == -9
    assert so.tdt_loss_fwd(*head[:3], 9, *head[4:], f, f, need, None) == -4
    # backward: grad_out required; grad_loss 4-byte aligned; workspace checked
    assert so.tdt_loss_bwd(*head, f, None, f, need, None) == -1
    assert so.tdt_loss_bwd(*head, ctypes.c_void_p(FAKE + 2), f, f, need, None) == -11
    assert so.tdt_loss_bwd(*head, None, f, None, need, None) == -1
    assert so.tdt_loss_bwd(*head, None, ctypes.c_void_p(FAKE + 4), f, need, None) == -13


def test_autograd_workspace_formula_matches_library(lib):
    from transducer_loss_asr_gb300.autograd import workspace_nbytes

    rng = __import__("random").Random(5)
    for _ in range(300):
        B, T, U1, nd = rng.randint(0, 20), rng.randint(1, 3000), rng.randint(1, 1300), \
            rng.randint(1, 32)
        if T + U1 > 65536:
            continue
        assert int(workspace_nbytes(B, T, U1, nd)) == lib.tdt_loss_workspace_size(
            [B, T, U1, nd + 5], nd)


def test_autograd_op_fake_shapes_and_cpu_rejection(lib):
    import torch

    from transducer_loss_asr_gb300 import autograd

    m = dict(device="meta")
    z = torch.empty(2, 5, 3, 13, **m)
    lab = torch.empty(2, 2, dtype=torch.long, **m)
    lens = torch.empty(2, dtype=torch.long, **m)
    for red, shape in (("mean", ()), ("none", (2,))):
        loss, ws = torch.ops.tdt_gb300.tdt_loss_forward(z, lab, lens, lens, [0, 1, 2], 6, 0.0, red)
        assert tuple(loss.shape) == shape and loss.dtype == torch.float32
        assert ws.numel() == lib.tdt_loss_workspace_size([2, 5, 3, 13], 3)
        g = torch.ops.tdt_gb300.tdt_loss_backward(loss, z, lab, lens, lens, ws, [0, 1, 2], 6,
                                                  0.0, red)
        assert g.shape == z.shape and g.dtype == z.dtype
    # the ops have CUDA kernels only: no silent CPU path
    with pytest.raises(NotImplementedError):
        autograd.tdt_loss(torch.zeros(2, 5, 3, 13), torch.zeros(2, 2, dtype=torch.long),
                          torch.full((2,), 5), torch.full((2,), 2), [0, 1, 2], 6)


def test_rnnt_entry_validates(lib):
    so = lib.lib
    f = ctypes.c_void_p(FAKE)

    def call(sizes, strides, dtype=0, blank=6, red=4, grad=f, sigma=0.0):
        return so.tdt_rnnt_loss_fwd_bwd(f, (ctypes.c_int64 * 4)(*sizes),
                                        (ctypes.c_int64 * 4)(*strides), dtype, f, f, f, blank,
                                        sigma, red, f, grad, None)

    ok_sizes, ok_strides = [2, 5, 3, 10], [150, 30, 10, 1]
    assert call([2, 5, 3, 0], ok_strides) == -2          # V >= 1
    assert call(ok_sizes, ok_strides, blank=10) == -6      # blank < V = 10 (no duration logits)
    assert call(ok_sizes, ok_strides, dtype=5) == -4
    assert call(ok_sizes, ok_strides, red=9) == -7
    assert call(ok_sizes, ok_strides, sigma=float("inf")) == -8
    assert call(ok_sizes, [150, 30, 10, 2]) == -3
    assert call(ok_sizes, ok_strides, grad=ctypes.c_void_p(FAKE + 4)) == -13


def test_greedy_decode_validates(lib):
    so = lib.lib
    f = ctypes.c_void_p(FAKE)
    durs = (ctypes.c_int32 * 3)(0, 1, 2)

    def call(sizes=(2, 5, 3, 10), strides=(150, 30, 10, 1), dtype=0, n_dur=3, blank=6,
             max_sym=4, logits=FAKE):
        return so.tdt_greedy_decode(ctypes.c_void_p(logits), (ctypes.c_int64 * 4)(*sizes),
                                    (ctypes.c_int64 * 4)(*strides), dtype, f, durs, n_dur,
                                    blank, max_sym, f, f, f, f, None)

    assert call(blank=7) == -6           # V = 10 - 3
    assert call(max_sym=0) == -2
    assert call(n_dur=0) == -5
    assert call(dtype=4) == -4
    assert call(sizes=(2, 0, 3, 10)) == -2
    assert call(strides=(150, 30, 10, 3)) == -3
    assert call(logits=FAKE + 2) == -11
    assert call(sizes=(0, 5, 3, 10)) == 0  # empty batch: nothing to do, nothing touched


def test_binding_import_fails_loudly_without_the_library(tmp_path):
    """No fallback: a copy of the package without libtdt_loss.so cannot load
    its binding; the error names the missing library and the build.  (The
    autograd op imports the binding in its device implementation, so its
    first CUDA call raises the same error.)"""
    import shutil
    import subprocess
    import sys

    src = os.path.join(ROOT, "transducer_loss_asr_gb300")
    shutil.copytree(src, tmp_path / "transducer_loss_asr_gb300",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    r = subprocess.run([sys.executable, "-c", "import transducer_loss_asr_gb300.binding"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libtdt_loss.so is not built" in r.stderr
