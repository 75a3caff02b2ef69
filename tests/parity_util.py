"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI binding and compare it with the fp64 oracle on the same bf16 inputs.

Tolerances (max absolute difference against the fp64 oracle, N(0,1) inputs):
O within 2e-2 and LSE within 1e-3."""
from __future__ import annotations

import numpy as np
import torch

import exact_attention_03_gb300 as fa
from oracle.naive import attention_head, to_f64

ATOL_O = 2e-2
ATOL_LSE = 1e-3


def run_gpu(q, k, v, causal, scale=None, stream=None):
    """q, k, v: CUDA bf16. Returns (O bf16, LSE fp32) and checks the device
    error word stayed clear."""
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, stream=stream)
    st, site = fa.last_device_error(stream)
    assert st == fa.FA_OK, f"device wait gave up: status {st} at site {site}"
    return o, lse


def compare_heads(q, k, v, o, lse, scale, causal, heads=None, rows=None):
    """Compares the GPU outputs with the oracle on the given (b, h) heads and,
    per head, query rows (None = all).  q/k/v/o/lse may live on any device.
    Returns (max |dO|, max |dLSE|, number of rows compared)."""
    B, H, Lq, D = q.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    worst_o = worst_l = 0.0
    n = 0
    for idx, (b, h) in enumerate(heads):
        r = None if rows is None else rows[idx]
        r_np = np.arange(Lq) if r is None else np.asarray(r, dtype=np.int64)
        qh = to_f64(q[b, h].cpu())
        kh = to_f64(k[b, h].cpu())
        vh = to_f64(v[b, h].cpu())
        o_ref, lse_ref = attention_head(qh, kh, vh, scale, causal=causal, rows=r_np)
        o_gpu = to_f64(o[b, h].cpu())[r_np]
        l_gpu = to_f64(lse[b, h].cpu())[r_np]
        assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(l_gpu))
        worst_o = max(worst_o, float(np.max(np.abs(o_gpu - o_ref))))
        worst_l = max(worst_l, float(np.max(np.abs(l_gpu - lse_ref))))
        n += len(r_np)
    return worst_o, worst_l, n


def assert_parity(q, k, v, causal, scale=None, heads=None, rows=None, stream=None):
    import math
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o, lse = run_gpu(q, k, v, causal, scale, stream=stream)
    torch.cuda.synchronize()
    do, dl, n = compare_heads(q, k, v, o, lse, scale, causal, heads=heads, rows=rows)
    assert do <= ATOL_O, f"max |dO| = {do:.3e} > {ATOL_O} over {n} rows"
    assert dl <= ATOL_LSE, f"max |dLSE| = {dl:.3e} > {ATOL_LSE} over {n} rows"
    return do, dl, n
