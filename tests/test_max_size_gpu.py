"""Forward and backward passes whose tensors hold more than 2^31 elements
each, so that every element offset past the first 2^31 must be computed in
64 bits (the TMA coordinates stay per head; the epilogues' O, LSE and
gradient addresses do not).  B = 1, L = 65536, and one head more than
2^31 / (L * D): the last head starts at element 2^31 or beyond.

* Forward: sampled rows (the first and last of the sequence and of a few
  tiles, plus random ones) of the first, a middle and the last head against
  the fp64 oracle, and at D = 128 the forward with dropout too.
* Backward (D = 128, causal): the oracle cannot hold a 65536-row head, so
  the first and last heads' outputs and gradients must equal, bit for bit,
  those of the same head computed alone (plain, and with dropout for head 0,
  whose index in the keep-bit counter is the same in both calls).

* Row softmax with rows * cols > 2^31, one case per kernel variant (a warp,
  shared memory or a CTA per row): sampled rows, the last ones included,
  against the fp64 oracle.

About 13 GB on the device for the forward cases, 35 GB for the backward and
17 GB for each softmax case."""
import math

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import Workload, make_inputs
from oracle import dropout as od
from oracle.naive import to_f64
from parity_util import ATOL_LSE, ATOL_O, compare_heads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
L = 65536


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _rows(seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 32767, 32768, L - 129, L - 128, L - 1]
    return np.unique(np.concatenate([fixed, rng.choice(L, 12, replace=False)]))


def _check():
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, f"device wait gave up: status {st} at site {site}"


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_forward_beyond_2_31_elements(D, causal):
    H = (1 << 31) // (L * D) + 1
    assert H * L * D > (1 << 31) and (H - 1) * L * D >= (1 << 31)
    w = Workload("max_size", 1, H, L, L, D, causal, seed=7)
    q, k, v = make_inputs(w, "cuda")
    o, lse = fa.forward(q, k, v, causal=causal)
    _check()
    torch.cuda.synchronize()
    heads = [(0, 0), (0, H // 2), (0, H - 1)]
    rows = [_rows(h) for _, h in heads]
    worst_o, worst_l, n = compare_heads(q, k, v, o, lse, w.scale, causal, heads=heads, rows=rows)
    print(f"D {D}: {n} rows, max|dO| {worst_o:.3e}, max|dLSE| {worst_l:.3e}")
    assert worst_o <= ATOL_O and worst_l <= ATOL_LSE
    if D == 128:
        p, seed, offset = 0.1, 99, 1
        del o, lse
        o, lse = fa.forward_dropout(q, k, v, p, seed, offset, causal=causal)
        _check()
        torch.cuda.synchronize()
        t = od.drop_threshold(p)
        for (b, h), r in zip(heads, rows):
            o_ref, lse_ref, _ = od.attention_dropout_rows(to_f64(q[b, h].cpu())[r], to_f64(k[b, h].cpu()),
                                                          to_f64(v[b, h].cpu()), w.scale, causal, r,
                                                          b * H + h, p, seed, offset)
            assert float(np.abs(to_f64(o[b, h].cpu())[r] - o_ref).max()) <= ATOL_O * 256 / (256 - t)
            assert float(np.abs(to_f64(lse[b, h].cpu())[r] - lse_ref).max()) <= ATOL_LSE
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_backward_beyond_2_31_elements_matches_each_head_alone():
    # the oracle cannot hold a 65536-row head in fp64; heads are independent
    # and the kernels deterministic, so a head's gradients inside the large
    # call must equal, bit for bit, those of the same head computed alone (a
    # wrong offset would read or write another head's rows)
    D, causal = 128, True
    H = (1 << 31) // (L * D) + 1
    w = Workload("max_size_bwd", 1, H, L, L, D, causal, seed=8)
    q, k, v = make_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(12)
    do = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    for p_drop in (None, 0.1):
        if p_drop is None:
            o, lse = fa.forward(q, k, v, causal=causal)
            grads = fa.backward(q, k, v, o, lse, do, causal=causal)
        else:
            o, lse = fa.forward_dropout(q, k, v, p_drop, 5, 0, causal=causal)
            grads = fa.backward_dropout(q, k, v, o, lse, do, p_drop, 5, 0, causal=causal)
        _check()
        for h in (0, H - 1):
            sl = lambda t: t[:, h:h + 1].contiguous()
            if p_drop is None:
                o1, lse1 = fa.forward(sl(q), sl(k), sl(v), causal=causal)
                g1 = fa.backward(sl(q), sl(k), sl(v), o1, lse1, sl(do), causal=causal)
            else:
                # the keep bits depend on the head's index in its call
                # (b*H + h), which a one-head call reproduces only for h = 0
                if h != 0:
                    continue
                o1, lse1 = fa.forward_dropout(sl(q), sl(k), sl(v), p_drop, 5, 0, causal=causal)
                g1 = fa.backward_dropout(sl(q), sl(k), sl(v), o1, lse1, sl(do), p_drop, 5, 0, causal=causal)
            _check()
            assert torch.equal(o1, sl(o)) and torch.equal(lse1, sl(lse)), (p_drop, h)
            for a, b in zip(g1, grads):
                assert torch.equal(a, sl(b)), (p_drop, h)
        del o, lse, grads
    del q, k, v, do
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cols", [1024, 8192, 32768])   # warp, shared-memory and CTA rows
def test_softmax_rows_beyond_2_31_elements(cols):
    from oracle.softmax import softmax_rows as oracle_softmax
    rows = (1 << 31) // cols + 1
    g = torch.Generator(device="cuda").manual_seed(cols)
    x = torch.randn(rows, cols, generator=g, device="cuda") * 4
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    pick = torch.tensor(sorted({0, 1, rows // 2, rows - 2, rows - 1}
                               | set(np.random.default_rng(cols).choice(rows, 8, replace=False).tolist())),
                        device="cuda")
    ry, rl = oracle_softmax(x[pick].cpu().numpy())
    assert np.abs(y[pick].cpu().numpy().astype(np.float64) - ry).max() <= 2e-6
    assert np.abs(lse[pick].cpu().numpy().astype(np.float64) - rl).max() <= 1e-5 * max(1.0, np.abs(rl).max())
    del x, y, lse
    torch.cuda.empty_cache()
