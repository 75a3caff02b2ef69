"""Seeded random shapes through the C ABI against the fp64 oracle, element by
element: the forward (head dims 64 and 128, causal or not, lengths that are
and are not multiples of the 128-row tiles, Lq != Lk, a custom scale, and
logits of several magnitudes) and the backward.  The shapes come from one
fixed generator, so a failure names a reproducible case; they complement the
hand-picked edge shapes of the other parity tests."""
import math
import random

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from oracle.backward import backward as oracle_backward
from parity_util import ATOL_LSE, ATOL_O, compare_heads, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _forward_cases(n=30, seed=2026):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        D = rng.choice((64, 128))
        causal = rng.random() < 0.5
        Lq = rng.choice((rng.randint(1, 160), rng.randint(100, 700), rng.randint(500, 1300)))
        Lk = Lq if causal else rng.choice((Lq, rng.randint(1, 1300)))
        if causal and Lq == 1:
            Lq = Lk = rng.randint(2, 300)
        B, H = rng.choice(((1, 1), (1, 3), (2, 2), (3, 1)))
        std = rng.choice((0.5, 1.0, 2.0, 3.0))
        scale = rng.choice((None, 0.05, 0.3))
        cases.append((i, B, H, Lq, Lk, D, causal, std, scale))
    return cases


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal,std,scale", _forward_cases())
def test_forward_random_shape(i, B, H, Lq, Lk, D, causal, std, scale):
    g = torch.Generator().manual_seed(1000 + i)
    q = (torch.randn(B, H, Lq, D, generator=g) * std).to(torch.bfloat16).cuda()
    k = (torch.randn(B, H, Lk, D, generator=g) * std).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16).cuda()
    s = 1.0 / math.sqrt(D) if scale is None else scale
    o, lse = run_gpu(q, k, v, causal, s)
    torch.cuda.synchronize()
    do, dl, n = compare_heads(q, k, v, o, lse, s, causal)
    assert do <= ATOL_O, f"case {i}: max |dO| = {do:.3e}"
    assert dl <= ATOL_LSE, f"case {i}: max |dLSE| = {dl:.3e}"


def _backward_cases(n=8, seed=77):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        D = rng.choice((64, 128))
        causal = rng.random() < 0.5
        Lq = rng.randint(30, 420)
        Lk = Lq if causal else rng.randint(30, 420)
        cases.append((i, rng.choice((1, 2)), rng.choice((1, 2)), Lq, Lk, D, causal))
    return cases


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal", _backward_cases())
def test_backward_random_shape(i, B, H, Lq, Lk, D, causal):
    g = torch.Generator().manual_seed(5000 + i)
    mk = lambda L: torch.randn(B, H, L, D, generator=g).to(torch.bfloat16).cuda()
    q, k, v, dout = mk(Lq), mk(Lk), mk(Lk), mk(Lq)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, dout, causal=causal, scale=scale)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    refs = oracle_backward(q.cpu(), k.cpu(), v.cpu(), dout.cpu(), scale, causal)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = float(np.abs(got.float().cpu().numpy().astype(np.float64) - ref).max())
        mag = float(np.abs(ref).max())
        assert err <= 2e-2 * max(1.0, mag), f"case {i} {name}: {err:.3e} (max |ref| {mag:.3e})"
