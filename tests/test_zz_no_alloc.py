"""The allocation-free single-query entry point against the regular one and
against the oracle.

fa_fwd_decode_noalloc exists for callers that cannot allocate device memory
while they run (an engine that plans all of its memory before serving, a
plugin held to a memory budget its host framework owns, a latency-critical
loop where growing a memory pool would stall); it keeps its split-K/V partial
results in a fixed array the library reserves on each GPU.  These tests call
it through the C ABI twice in a row (the array keeps the previous call's
contents, which must not leak into the next result) and compare each result
with fa_fwd on the same inputs (bit for bit where both use the same number of
key splits) and with the fp64 oracle; they exercise the Python wrapper and
its argument checks, and check, in a fresh process, that repeated calls of
several sizes leave the device's free memory unchanged.
This file is collected last on purpose.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import Workload, make_inputs
from parity_util import ATOL_LSE, ATOL_O, compare_heads

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()


def _raw_noalloc(q, k, v, o, lse, scale):
    B, H, _, D = q.shape
    return fa.load().fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), B, H, k.shape[2], D, scale,
                                           torch.cuda.current_stream().cuda_stream)


def _same_splits(B, H, Lk, D):
    """True when fa_fwd and the no-alloc call split the keys the same way."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    n = fa.decode_num_splits(B * H, Lk, sms)
    cap = fa.load().fa_decode_noalloc_max_floats() // (B * H * (D + 2))
    return n <= cap


@pytest.mark.parametrize("B,H,Lk,D", [
    (2, 8, 50000, 128),     # the regular split count fits in the array
    (8, 128, 16384, 128),   # the array caps the split count below fa_fwd's
    (3, 5, 777, 64),
])
def test_noalloc_matches_fa_fwd_and_oracle_twice(B, H, Lk, D):
    w = Workload("noalloc", B, H, 1, Lk, D, False, seed=31)
    q, k, v = make_inputs(w, "cuda")
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref = fa.forward(q, k, v, causal=False)
    assert fa.last_device_error()[0] == fa.FA_OK
    exact = _same_splits(B, H, Lk, D)
    # the oracle on every head, or on 40 sampled heads of the large case
    heads = [(b, h) for b in range(B) for h in range(H)]
    if len(heads) > 64:
        heads = [heads[i] for i in np.random.default_rng(0).choice(len(heads), 40, replace=False)]
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _raw_noalloc(q, k, v, o, lse, scale) == fa.FA_OK
        assert fa.last_device_error()[0] == fa.FA_OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        if exact:
            assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
        else:
            assert (o.float() - o_ref.float()).abs().max().item() <= ATOL_O
            assert (lse - lse_ref).abs().max().item() <= ATOL_LSE
        d_o, d_l, _ = compare_heads(q, k, v, o, lse, scale, False, heads=heads)
        assert d_o <= ATOL_O and d_l <= ATOL_LSE, (d_o, d_l)


def test_python_wrapper_matches_and_checks_shapes():
    w = Workload("noalloc_py", 2, 4, 1, 3000, 128, False, seed=32)
    q, k, v = make_inputs(w, "cuda")
    o_ref, lse_ref = fa.forward(q, k, v, causal=False)
    out = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    o, l = fa.decode_noalloc(q, k, v, out=out, lse=lse)
    assert o is out and l is lse
    assert torch.equal(o, o_ref) and torch.equal(l, lse_ref)
    bad_k = [k[:, :3].contiguous(),                 # fewer heads
             k[:1].contiguous(),                    # another batch size
             torch.zeros(2, 4, 3000, 64, dtype=torch.bfloat16, device="cuda")]  # another D
    for kk in bad_k:
        with pytest.raises(ValueError):
            fa.decode_noalloc(q, kk, kk.clone())
    with pytest.raises(ValueError):
        fa.decode_noalloc(q, k, v[:, :, :2000].contiguous())   # v shaped unlike k
    with pytest.raises(ValueError):
        fa.decode_noalloc(q, k, v, out=torch.empty(2, 4, 1, 64, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.decode_noalloc(q, k, v, lse=torch.empty(3, dtype=torch.float32, device="cuda"))


_NO_GROWTH = r"""
import json, math, torch
import exact_attention_03_gb300 as fa
from exact_attention_03_gb300.inputs import Workload, make_inputs
lib = fa.load()
probs = []
for (B, H, Lk) in ((1, 1, 64), (4, 32, 20000), (8, 128, 16384)):
    q, k, v = make_inputs(Workload("g", B, H, 1, Lk, 128, False, seed=33), "cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
    probs.append((q, k, v, o, lse))
def call(p):
    q, k, v, o, lse = p
    B, H, _, D = q.shape
    return lib.fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, k.shape[2], D, 1 / math.sqrt(D),
                                     torch.cuda.current_stream().cuda_stream)
st = [call(probs[0])]          # loads the kernels and looks up the array's address
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    st += [call(p) for p in probs]
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
print(json.dumps({"status": st, "free0": free0, "free1": free1}))
"""


def test_repeated_calls_leave_free_memory_unchanged():
    # A fresh process in which fa_fwd never runs (so the library's workspace
    # pool does not exist): after one small call, calls that would need far
    # more workspace, if they allocated any, must not change the free memory.
    r = subprocess.run([sys.executable, "-c", _NO_GROWTH], cwd=ROOT, capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, PYTHONPATH=ROOT))
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert all(s == fa.FA_OK for s in res["status"]), res
    assert res["free0"] == res["free1"], res


def test_noalloc_rejects_what_does_not_fit():
    cap = fa.load().fa_decode_noalloc_max_floats()
    D = 128
    H = cap // (D + 2) + 1  # one head too many for a single split
    a = 1 << 20
    st = fa.load().fa_fwd_decode_noalloc(a, a, a, a, a, 1, H, 1000, D, 0.1, None)
    assert st == fa.FA_ERR_UNSUPPORTED
