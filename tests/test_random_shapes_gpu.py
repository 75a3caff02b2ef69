"""Seeded random shapes through the C ABI against the fp64 oracles, element by
element: the forward (head dims 64 and 128, causal or not, lengths that are
and are not multiples of the 128-row tiles, Lq != Lk, a custom scale, and
logits of several magnitudes), the backward, the forward with dropout
(random p, 64-bit seeds and offsets) and its backward, and the paged decode (random page
sizes, lengths, empty sequences, page tables); and forward cases with many
heads, whose grids run several waves and walk the heads in L2-sized groups
with a ragged last group, checked on sampled heads.  The shapes come from one
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


def _many_head_cases(n=8, seed=4254):
    # grids of several waves, heads walked in L2-sized groups with a ragged last
    # group (24 MB of K/V per group: 8 to 64 heads at these lengths)
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        D = rng.choice((64, 128))
        causal = rng.random() < 0.5
        Lq = rng.randint(200, 1600)
        Lk = Lq if causal else rng.choice((Lq, rng.randint(150, 1600)))
        B = rng.choice((2, 3, 4))
        H = rng.choice((5, 12, 17, 24))
        cases.append((i, B, H, Lq, Lk, D, causal))
    return cases


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal", _many_head_cases())
def test_forward_many_heads(i, B, H, Lq, Lk, D, causal):
    g = torch.Generator().manual_seed(5000 + i)
    q = torch.randn(B, H, Lq, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16).cuda()
    s = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, s)
    torch.cuda.synchronize()
    # the first and last heads, one in the middle and a random one; all rows of
    # the first, sampled rows (tile boundaries and the last row) of the others
    rng = random.Random(i)
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 2), (rng.randrange(B), rng.randrange(H))]
    rows = [None] + [np.unique(np.clip(np.array([0, 127, 128, Lq // 2, Lq - 1] +
                                                 [rng.randrange(Lq) for _ in range(40)]), 0, Lq - 1))] * 3
    do, dl, n = compare_heads(q, k, v, o, lse, s, causal, heads=heads, rows=rows)
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


def _dropout_cases(n=10, seed=31):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        D = rng.choice((64, 128))
        causal = rng.random() < 0.5
        Lq = rng.randint(1, 600)
        Lk = Lq if causal else rng.randint(1, 600)
        if causal and Lq == 1:
            Lq = Lk = 2
        p = rng.choice((0.0, 0.05, 0.2, 0.5, 0.9))
        seed64 = rng.getrandbits(64)
        offset = rng.getrandbits(32)
        cases.append((i, rng.choice((1, 2)), rng.choice((1, 3)), Lq, Lk, D, causal, p, seed64, offset))
    return cases


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal,p,seed64,offset", _dropout_cases())
def test_dropout_random_shape(i, B, H, Lq, Lk, D, causal, p, seed64, offset):
    from oracle import dropout as od
    from oracle.naive import to_f64
    g = torch.Generator().manual_seed(7000 + i)
    q = torch.randn(B, H, Lq, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16).cuda()
    o, lse = fa.forward_dropout(q, k, v, p, seed64, offset, causal=causal)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    t = od.drop_threshold(p)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for h in range(H):
            ro, rl, _ = od.attention_dropout_rows(to_f64(q[b, h].cpu()), to_f64(k[b, h].cpu()),
                                                  to_f64(v[b, h].cpu()), scale, causal, np.arange(Lq),
                                                  b * H + h, p, seed64, offset)
            d_o = float(np.abs(to_f64(o[b, h].cpu()) - ro).max())
            d_l = float(np.abs(to_f64(lse[b, h].cpu()) - rl).max())
            assert d_o <= ATOL_O * 256 / (256 - t), f"case {i}: max |dO| = {d_o:.3e}"
            assert d_l <= ATOL_LSE, f"case {i}: max |dLSE| = {d_l:.3e}"


def _dropout_backward_cases(n=8, seed=91):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        D = rng.choice((64, 128))
        causal = rng.random() < 0.5
        Lq = rng.randint(20, 420)
        Lk = Lq if causal else rng.randint(20, 420)
        p = rng.choice((0.05, 0.2, 0.5, 0.9))
        cases.append((i, rng.choice((1, 2)), rng.choice((1, 2)), Lq, Lk, D, causal, p, rng.getrandbits(64),
                      rng.getrandbits(32)))
    return cases


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal,p,seed64,offset", _dropout_backward_cases())
def test_dropout_backward_random_shape(i, B, H, Lq, Lk, D, causal, p, seed64, offset):
    from oracle import dropout as od
    from oracle.naive import to_f64
    g = torch.Generator().manual_seed(9000 + i)
    mk = lambda L: torch.randn(B, H, L, D, generator=g).to(torch.bfloat16).cuda()
    q, k, v, dout = mk(Lq), mk(Lk), mk(Lk), mk(Lq)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward_dropout(q, k, v, p, seed64, offset, causal=causal)
    dq, dk, dv = fa.backward_dropout(q, k, v, o, lse, dout, p, seed64, offset, causal=causal)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    refs = od.backward_dropout(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), to_f64(dout.cpu()), scale,
                               causal, p, seed64, offset)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = float(np.abs(to_f64(got.cpu()) - ref).max())
        mag = float(np.abs(ref).max())
        assert err <= 2e-2 * max(1.0, mag), f"case {i} {name}: {err:.3e} (max |ref| {mag:.3e})"


def _paged_cases(n=6, seed=53):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        page = rng.choice((1, 4, 16, 64, 256))
        max_pages = rng.randint(1, max(1, 3000 // page))
        B = rng.randint(1, 5)
        lengths = tuple(rng.randint(0, max_pages * page) for _ in range(B))
        cases.append((i, B, rng.choice((1, 4)), rng.choice((64, 128)), page, max_pages, lengths))
    return cases


@pytest.mark.parametrize("i,B,H,D,page,max_pages,lengths", _paged_cases())
def test_paged_random_shape(i, B, H, D, page, max_pages, lengths):
    from exact_attention_03_gb300.inputs import PagedWorkload, make_paged_inputs
    from oracle.paged import decode_paged as oracle_paged
    w = PagedWorkload(f"r{i}", B, H, D, page, max_pages * page, 300 + i, lengths=lengths)
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    o, lse = fa.decode_paged(q, kc, vc, bt, lens, scale=w.scale)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    ro, rl = oracle_paged(q.cpu(), kc.cpu(), vc.cpu(), bt.cpu(), lens.cpu(), w.scale)
    go = o.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(gl), empty)
    assert np.all(go[empty] == 0)
    assert float(np.abs(go - ro).max()) <= ATOL_O
    if (~empty).any():
        assert float(np.abs(gl[~empty] - rl[~empty]).max()) <= ATOL_LSE
