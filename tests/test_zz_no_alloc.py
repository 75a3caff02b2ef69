"""The allocation-free single-query entry point against the regular one.

fa_fwd_decode_noalloc exists for callers that cannot allocate device memory
while they run; it keeps its split-K/V partial results in a fixed array the
library reserves at load time.  These tests call it through the C ABI twice
in a row (the array keeps the previous call's contents, which must not leak
into the next result) and compare each result with fa_fwd on the same inputs.
This file is collected last on purpose.
"""
import math

import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import Workload, make_inputs
from parity_util import ATOL_LSE, ATOL_O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()


def _raw_noalloc(q, k, v, o, lse, scale):
    B, H, _, D = q.shape
    return fa.load().fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), B, H, k.shape[2], D, scale,
                                           torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,Lk,D", [
    (2, 8, 50000, 128),     # the regular split count fits in the array
    (8, 128, 16384, 128),   # the array caps the split count below fa_fwd's
    (3, 5, 777, 64),
])
def test_noalloc_matches_fa_fwd_twice(B, H, Lk, D):
    w = Workload("noalloc", B, H, 1, Lk, D, False, seed=31)
    q, k, v = make_inputs(w, "cuda")
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref = fa.forward(q, k, v, causal=False)
    assert fa.last_device_error()[0] == fa.FA_OK
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _raw_noalloc(q, k, v, o, lse, scale) == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - o_ref.float()).abs().max().item() <= ATOL_O
        assert (lse - lse_ref).abs().max().item() <= ATOL_LSE


def test_noalloc_rejects_what_does_not_fit():
    cap = fa.load().fa_decode_noalloc_max_floats()
    D = 128
    H = cap // (D + 2) + 1  # one head too many for a single split
    a = 1 << 20
    st = fa.load().fa_fwd_decode_noalloc(a, a, a, a, a, 1, H, 1000, D, 0.1, None)
    assert st == fa.FA_ERR_UNSUPPORTED
