"""GPU parity of the backward pass (fa_bwd through the C ABI, on top of our
own forward) with the fp64 oracle oracle.backward, element by element: head
dims 64 and 128, causal and not, several key and query tiles, ragged tails,
Lq != Lk without the mask, a single tile, and larger logits.

Tolerance: the gradients come out in bf16, and P and dS enter the tensor-core
products rounded to bf16 (relative 2^-9 each), as does the forward's O that
Dr = rowsum(dO * O) uses; each gradient element is a sum of such products, so
the bound is relative to the tensor's largest magnitude:
max|d - d_ref| <= 2e-2 * max(1, max|d_ref|)."""
import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from oracle.backward import backward as oracle_backward

pytestmark = pytest.mark.gpu
RTOL_GRAD = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _inputs(B, H, Lq, Lk, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda L, s=1.0: (torch.randn(B, H, L, D, generator=g) * s).to(torch.bfloat16).cuda()
    return mk(Lq, std), mk(Lk, std), mk(Lk), mk(Lq)


def _errors(q, k, v, do, causal, scale=None):
    D = q.shape[-1]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    refs = oracle_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, causal)
    out = {}
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        g = got.float().cpu().numpy().astype(np.float64)
        out[name] = (np.abs(g - ref).max(), np.abs(ref).max())
    return out


CASES = [
    (1, 2, 256, 256, 64, False),
    (1, 2, 256, 256, 128, False),
    (1, 2, 384, 384, 64, True),
    (1, 2, 300, 300, 128, True),
    (2, 1, 200, 333, 128, False),
    (1, 3, 128, 128, 64, True),
    (1, 1, 77, 77, 64, False),
]


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", CASES)
def test_backward_parity(B, H, Lq, Lk, D, causal):
    q, k, v, do = _inputs(B, H, Lq, Lk, D, seed=Lq + D + causal)
    for name, (err, mag) in _errors(q, k, v, do, causal).items():
        print(f"{name}: max err {err:.3e}  max |ref| {mag:.3e}")
        assert err <= RTOL_GRAD * max(1.0, mag), (name, err, mag)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_backward_sharp_logits(D, causal):
    q, k, v, do = _inputs(1, 2, 512, 512, D, seed=99, std=3.0)
    for name, (err, mag) in _errors(q, k, v, do, causal).items():
        print(f"{name}: max err {err:.3e}  max |ref| {mag:.3e}")
        assert err <= RTOL_GRAD * max(1.0, mag), (name, err, mag)
