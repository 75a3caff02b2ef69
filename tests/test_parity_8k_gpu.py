"""Oracle parity of the backward pass and of the forward with dropout at the
sizes the benchmark times them at, in the benchmark's launch configuration.

* Backward (fa_bwd), causal B2 H32 L8192 D128 with the benchmark's dO (a CUDA
  generator seeded 11): the whole problem runs on the GPU, then whole heads
  are compared element by element with oracle.backward.backward_head: head 0
  (in the first L2 head group of both backward kernels: groups of 6 heads at
  4 MB of Q+dO or K+V per head) , head 37 (a middle full group) and head 63
  (in the 4-head remainder group).  Every head has 64 key tiles and 64 query
  tiles, so the long loops and the multi-group grid order meet the oracle.
* Forward with dropout (fa_fwd_dropout, p = 0.1, seed 1234, offset 0) on the
  causal 8K D128 workload and on the sweep's L = 8192 D64 workload (B4 H8):
  sampled query rows (the first and last row of the sequence and of a few
  tiles, plus random rows) of sampled heads against
  oracle.dropout.attention_dropout_rows, which draws the keep bits on the
  CPU from the contract.

Tolerances as in the smaller tests: gradients within 2e-2 * max(1, max|ref|)
per tensor; O within 2e-2 * 256 / (256 - t), LSE within 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import WORKLOADS, Workload, make_inputs
from oracle import dropout as od
from oracle.backward import backward_head
from oracle.naive import to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
RTOL_GRAD = 2e-2
ATOL_O = 2e-2
ATOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _check():
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, f"device wait gave up: status {st} at site {site}"


def test_backward_causal_l8k_d128_whole_heads():
    w = WORKLOADS["causal_l8k_d128"]
    dev = torch.device("cuda")
    q, k, v = make_inputs(w, dev)
    g = torch.Generator(device=dev).manual_seed(11)
    do = torch.randn(q.shape, generator=g, device=dev).to(torch.bfloat16)
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    _check()
    torch.cuda.synchronize()
    for bh in (0, 37, 63):
        b, h = divmod(bh, w.H)
        refs = backward_head(to_f64(q[b, h].cpu()), to_f64(k[b, h].cpu()), to_f64(v[b, h].cpu()),
                             to_f64(do[b, h].cpu()), w.scale, causal=True)
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            err = float(np.abs(to_f64(got[b, h].cpu()) - ref).max())
            mag = float(np.abs(ref).max())
            print(f"head {bh} {name}: max err {err:.3e}  max |ref| {mag:.3e}")
            assert err <= RTOL_GRAD * max(1.0, mag), (bh, name, err, mag)
        del refs


def _sample_rows(L, n_random, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 255, 4095, 4096, L - 129, L - 128, L - 1]
    return np.unique(np.concatenate([fixed, rng.choice(L, n_random, replace=False)]))


@pytest.mark.parametrize("name,heads", [
    ("causal_l8k_d128", (0, 31, 37, 63)),
    ("sweep_l8192_d64", (0, 13, 31)),
])
def test_dropout_l8k_sampled_rows(name, heads):
    if name == "causal_l8k_d128":
        w = WORKLOADS[name]
    else:
        w = Workload("sweep_8192", 4, 8, 8192, 8192, 64, False, seed=1)
    dev = torch.device("cuda")
    q, k, v = make_inputs(w, dev)
    p, seed, offset = 0.1, 1234, 0
    o, lse = fa.forward_dropout(q, k, v, p, seed, offset, causal=w.causal)
    _check()
    torch.cuda.synchronize()
    t = od.drop_threshold(p)
    worst_o = worst_l = 0.0
    for bh in heads:
        b, h = divmod(bh, w.H)
        rows = _sample_rows(w.Lq, 40, seed=bh)
        qh = to_f64(q[b, h].cpu())
        o_ref, lse_ref, _ = od.attention_dropout_rows(qh[rows], to_f64(k[b, h].cpu()),
                                                      to_f64(v[b, h].cpu()), w.scale, w.causal, rows,
                                                      bh, p, seed, offset)
        worst_o = max(worst_o, float(np.abs(to_f64(o[b, h].cpu())[rows] - o_ref).max()))
        worst_l = max(worst_l, float(np.abs(to_f64(lse[b, h].cpu())[rows] - lse_ref).max()))
    print(f"{name}: max|dO| {worst_o:.3e}  max|dLSE| {worst_l:.3e}")
    assert worst_o <= ATOL_O * 256 / (256 - t)
    assert worst_l <= ATOL_LSE
