"""Greedy TDT decoding on the GPU (tdt_greedy_decode) against the decoding
oracle: token, frame and duration sequences must agree exactly (integer
results; the argmax compares the same exactly converted values)."""
import numpy as np
import pytest
import torch

from oracle.decode import tdt_greedy_decode as oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transducer_loss_asr_gb300 import binding as b

    return b


def _compare(binding, z, tl, durs, blank, max_symbols):
    n, tok, frm, dur = binding.tdt_greedy_decode(z, tl, durs, blank, max_symbols)
    torch.cuda.synchronize()
    rn, rt, rf, rd = oracle_decode(z.float().cpu().numpy(), tl.cpu().numpy(), durs, blank,
                                   max_symbols)
    np.testing.assert_array_equal(n.cpu().numpy(), rn)
    np.testing.assert_array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_array_equal(frm.cpu().numpy(), rf)
    np.testing.assert_array_equal(dur.cpu().numpy(), rd)
    return rn


def test_planted_path(binding):
    V, durs, blank = 8, [0, 1, 2, 3, 4], 7
    g = torch.Generator().manual_seed(1)
    z = torch.rand(1, 7, 5, V + 5, generator=g) * 2 - 1
    for (t, u, k, di) in [(0, 0, 3, 0), (0, 1, 5, 2), (2, 2, blank, 1), (3, 2, 1, 3),
                          (6, 3, blank, 0)]:
        z[0, t, u, k] = 5.0
        z[0, t, u, V + di] = 5.0
    n = _compare(binding, z.cuda(), torch.tensor([7]).cuda(), durs, blank, 10)
    assert n[0] == 3


@pytest.mark.parametrize("dtype,max_symbols,base", [(torch.float32, 10, None),
                                                    (torch.float32, 1, 140),
                                                    (torch.bfloat16, 3, None),
                                                    (torch.float16, 2, None)])
def test_random_logits(binding, dtype, max_symbols, base):
    g = torch.Generator(device="cuda").manual_seed(17)
    B, T, U, V, durs, blank = 6, 50, 20, 120, [0, 1, 2, 4], 0
    W = base or V + len(durs)
    z = torch.randn(B, T, U + 1, W, generator=g, device="cuda")
    z[..., blank] += 1.0   # blank often wins
    z[..., V + 0] += 0.7   # duration 0 often wins: exercises the symbol guard
    z = z.to(dtype)[..., : V + len(durs)]
    tl = torch.tensor([50, 1, 37, 0, 50, 12], device="cuda")  # T_b = 0: nothing decoded
    n = _compare(binding, z, tl, durs, blank, max_symbols)
    assert n[3] == 0 and n.max() > 0


def test_bf16_ties(binding):
    # a coarse grid of values makes equal maxima common: ties go to the first index
    g = torch.Generator(device="cuda").manual_seed(5)
    z = torch.randint(-2, 3, (4, 30, 9, 37), generator=g, device="cuda").to(torch.bfloat16)
    tl = torch.full((4,), 30, device="cuda")
    _compare(binding, z, tl, [0, 1, 3], 33, 4)


def test_parakeet_size(binding):
    from transducer_loss_asr_gb300.workloads import make_inputs

    inp = make_inputs("parakeet", device="cuda")
    _compare(binding, inp["logits"], inp["logit_lens"], inp["durations"], inp["blank"], 10)
