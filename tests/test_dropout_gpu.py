"""GPU parity of attention with dropout (fa_fwd_dropout through the C ABI)
with the fp64 oracle oracle.dropout, which draws the same Philox bits on the
CPU from the contract's definition:

* the keep mask itself, bit for bit: with v = identity (Lk = D) the output
  row is the dropped, rescaled weight row, so every dropped weight reads 0;
* O and LSE element by element for head dims 64 and 128, causal and not,
  ragged lengths, a single query row, 64-bit seeds and offsets;
* LSE is exactly the plain forward's, and p = 0 gives the plain forward's O.

Tolerance: O within 2e-2 * 256 / (256 - t) (the rescale multiplies the
values and their bf16 rounding alike), LSE within 1e-3."""
import math

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from oracle import dropout as od
from oracle.naive import to_f64

pytestmark = pytest.mark.gpu
ATOL_O = 2e-2
ATOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _inputs(B, H, Lq, Lk, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda L, s: (torch.randn(B, H, L, D, generator=g) * s).to(torch.bfloat16).cuda()
    return mk(Lq, std), mk(Lk, std), mk(Lk, 1.0)


def _run(q, k, v, p, seed, offset, causal):
    o, lse = fa.forward_dropout(q, k, v, p, seed, offset, causal=causal)
    st, site = fa.last_device_error(None)
    assert st == fa.FA_OK, f"device wait gave up: status {st} at site {site}"
    torch.cuda.synchronize()
    return o, lse


def _compare(q, k, v, o, lse, p, seed, offset, causal):
    B, H, Lq, D = q.shape
    scale = 1.0 / math.sqrt(D)
    t = od.drop_threshold(p)
    worst_o = worst_l = 0.0
    rows = np.arange(Lq)
    for b in range(B):
        for h in range(H):
            o_ref, lse_ref, _ = od.attention_dropout_rows(to_f64(q[b, h].cpu()), to_f64(k[b, h].cpu()),
                                                          to_f64(v[b, h].cpu()), scale, causal, rows, b * H + h,
                                                          p, seed, offset)
            worst_o = max(worst_o, float(np.abs(to_f64(o[b, h].cpu()) - o_ref).max()))
            worst_l = max(worst_l, float(np.abs(to_f64(lse[b, h].cpu()) - lse_ref).max()))
    assert worst_o <= ATOL_O * 256 / (256 - t), f"max |dO| = {worst_o:.3e}"
    assert worst_l <= ATOL_LSE, f"max |dLSE| = {worst_l:.3e}"


@pytest.mark.parametrize("D,causal,Lq", [(64, False, 300), (64, True, 64), (128, False, 200), (128, True, 128)])
@pytest.mark.parametrize("p", [0.1, 0.5, 0.8])
def test_keep_mask_bit_exact(D, causal, Lq, p):
    # v = identity over the Lk = D keys: O[i, j] = w_ij z_ij 256 / (256 - t)
    B, H, Lk = 1, 2, D
    if causal:
        Lq = Lk
    g = torch.Generator().manual_seed(7)
    q = (torch.randn(B, H, Lq, D, generator=g) * 0.3).to(torch.bfloat16).cuda()
    k = (torch.randn(B, H, Lk, D, generator=g) * 0.3).to(torch.bfloat16).cuda()
    v = torch.eye(D, dtype=torch.bfloat16).expand(B, H, Lk, D).contiguous().cuda()
    seed, offset = 0x1234_5678_9ABC_DEF0, 3
    o, lse = _run(q, k, v, p, seed, offset, causal)
    t = od.drop_threshold(p)
    for h in range(H):
        z = od.keep_mask(h, np.arange(Lq), Lk, t, seed, offset)
        visible = np.ones((Lq, Lk), dtype=bool)
        if causal:
            visible = np.tril(visible)
        nonzero = to_f64(o[0, h].cpu())[:, :Lk] != 0
        # small logits: every visible weight is far from underflow, so a zero is a drop
        assert np.array_equal(nonzero[visible], z[visible])
        assert not nonzero[~visible].any()
    _compare(q, k, v, o, lse, p, seed, offset, causal)


@pytest.mark.parametrize("D,causal,Lq,Lk", [
    (64, False, 200, 384),
    (128, False, 130, 520),
    (128, True, 384, 384),
    (64, True, 448, 448),
])
def test_keep_mask_bit_exact_past_the_first_key_tile(D, causal, Lq, Lk):
    # One call per block of D keys, with v = the identity on that block and
    # zero elsewhere: O[i, c] = w_(i, blk*D + c) z_(i, blk*D + c) 256 / (256 - t),
    # so every key tile (counter words j div 16 up to Lk / 16) is read bit by bit.
    B, H = 1, 2
    p, seed, offset = 0.1, 0xFEDC_BA98_7654_3210, 77
    g = torch.Generator().manual_seed(8)
    q = (torch.randn(B, H, Lq, D, generator=g) * 0.3).to(torch.bfloat16).cuda()
    k = (torch.randn(B, H, Lk, D, generator=g) * 0.3).to(torch.bfloat16).cuda()
    t = od.drop_threshold(p)
    z = [od.keep_mask(h, np.arange(Lq), Lk, t, seed, offset) for h in range(H)]
    visible = np.tril(np.ones((Lq, Lk), dtype=bool)) if causal else np.ones((Lq, Lk), dtype=bool)
    seen = np.zeros((H, Lq, Lk), dtype=bool)
    for blk in range((Lk + D - 1) // D):
        lo, hi = blk * D, min(Lk, (blk + 1) * D)
        v = torch.zeros(B, H, Lk, D, dtype=torch.bfloat16)
        v[:, :, lo:hi, :hi - lo] = torch.eye(hi - lo, dtype=torch.bfloat16)
        o, _ = _run(q, k, v.cuda(), p, seed, offset, causal)
        for h in range(H):
            nonzero = to_f64(o[0, h].cpu())[:, :hi - lo] != 0
            vis = visible[:, lo:hi]
            assert np.array_equal(nonzero[vis], z[h][:, lo:hi][vis]), (blk, h)
            assert not nonzero[~vis].any()
            seen[h, :, lo:hi] = True
    assert seen.all()


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [
    (1, 2, 300, 300, 128, True),
    (2, 1, 257, 384, 64, False),
    (1, 2, 200, 520, 128, False),
    (1, 1, 1, 700, 128, False),      # a single query row (runs on the prefill kernel)
    (1, 1, 1, 256, 64, False),
    (1, 3, 129, 129, 64, True),
])
def test_parity_with_oracle(B, H, Lq, Lk, D, causal):
    q, k, v = _inputs(B, H, Lq, Lk, D, seed=B * 1000 + Lq + Lk)
    for p, seed, offset in ((0.1, 5, 0), (0.3, (1 << 40) + 17, 123456)):
        o, lse = _run(q, k, v, p, seed, offset, causal)
        _compare(q, k, v, o, lse, p, seed, offset, causal)


@pytest.mark.parametrize("D", [64, 128])
def test_lse_and_p_zero_match_the_plain_forward(D):
    q, k, v = _inputs(2, 2, 384, 384, D, seed=11)
    o0, lse0 = fa.forward(q, k, v, causal=True)
    o1, lse1 = _run(q, k, v, 0.25, 99, 1, True)
    assert torch.equal(lse0, lse1)
    assert not torch.equal(o0, o1)
    o2, lse2 = _run(q, k, v, 0.0, 99, 1, True)
    assert torch.equal(lse0, lse2)
    assert float((o2.float() - o0.float()).abs().max()) <= 1e-2


def test_seed_and_offset_select_different_bits():
    q, k, v = _inputs(1, 1, 256, 256, 128, seed=3)
    outs = [_run(q, k, v, 0.5, s, off, False)[0] for s, off in ((1, 0), (2, 0), (1, 1), (1 | (1 << 32), 0))]
    for a in range(len(outs)):
        for b in range(a + 1, len(outs)):
            assert not torch.equal(outs[a], outs[b])
    # and the same (seed, offset) reproduces exactly
    assert torch.equal(outs[0], _run(q, k, v, 0.5, 1, 0, False)[0])
