"""GPU parity of the backward pass of attention with dropout (fa_bwd_dropout
through the C ABI, after fa_fwd_dropout) with the fp64 oracle
oracle.dropout.backward_dropout, which draws the same Philox keep bits on the
CPU from the contract's definition:

* the keep bits each kernel draws, bit for bit.  With q, k and v whose rows
  are unit vectors (row i is e_(i mod D)), every weight is far from
  underflow, and the gradients read the dropped weights out one by one:
  - dO = e_(i mod D) on one block of D query rows and 0 elsewhere:
    dv[j, c] = s w z at (row qb D + c, key j), so the key-tile kernel's
    dropped weights of that block are exactly its zeros;
  - o = 0 passed in (so rowsum(dO * O) = 0) and random nonzero dO: the
    weight gradients are dA = s w z * (dO v^T), and
    dq[i, c] = scale dA[i, kb D + c] when v is zero outside key block kb
    (the query-tile kernel's bits), dk[j, c] = scale dA[qb D + c, j] when
    dO is zero outside query block qb (the key-tile kernel's bits again,
    through the dS path);
* dq, dk, dv element by element for head dims 64 and 128, causal and not,
  ragged lengths, several key and query tiles, p = 0.1, 0.5, 0.8 (and 0.99),
  64-bit seeds and offsets, a single query row or key;
* p = 0 gives fa_bwd's gradients bit for bit;
* two whole heads of the causal L = 8192 D = 128 workload (slow).

Tolerance as for fa_bwd: max|d - d_ref| <= 2e-2 * max(1, max|d_ref|) per
tensor (the kept weights' rescale multiplies values and their rounding
alike)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs
from oracle import dropout as od
from oracle.naive import to_f64

pytestmark = pytest.mark.gpu
RTOL_GRAD = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _check():
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, f"device wait gave up: status {st} at site {site}"


def _inputs(B, H, Lq, Lk, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda L, s=1.0: (torch.randn(B, H, L, D, generator=g) * s).to(torch.bfloat16).cuda()
    return mk(Lq, std), mk(Lk, std), mk(Lk), mk(Lq)


def _grads(q, k, v, do, p, seed, offset, causal):
    o, lse = fa.forward_dropout(q, k, v, p, seed, offset, causal=causal)
    dq, dk, dv = fa.backward_dropout(q, k, v, o, lse, do, p, seed, offset, causal=causal)
    _check()
    torch.cuda.synchronize()
    return dq, dk, dv


def _compare(q, k, v, do, got, p, seed, offset, causal):
    scale = 1.0 / math.sqrt(q.shape[-1])
    refs = od.backward_dropout(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), to_f64(do.cpu()), scale,
                               causal, p, seed, offset)
    for name, g, ref in zip(("dq", "dk", "dv"), got, refs):
        err = float(np.abs(to_f64(g.cpu()) - ref).max())
        mag = float(np.abs(ref).max())
        print(f"p {p} {name}: max err {err:.3e}  max |ref| {mag:.3e}")
        assert err <= RTOL_GRAD * max(1.0, mag), (name, p, err, mag)


CASES = [
    (1, 2, 256, 256, 64, False),
    (1, 2, 256, 256, 128, False),
    (1, 2, 384, 384, 64, True),
    (1, 2, 300, 300, 128, True),
    (2, 1, 200, 333, 128, False),
    (1, 3, 129, 129, 64, True),
    (1, 1, 77, 77, 64, False),
]


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", CASES)
def test_parity_with_oracle(B, H, Lq, Lk, D, causal):
    q, k, v, do = _inputs(B, H, Lq, Lk, D, seed=3 * Lq + D + causal)
    for p, seed, offset in ((0.1, 5, 0), (0.5, (1 << 40) + 17, 123456), (0.8, 0xFFFF_FFFF_FFFF_FFFF, 0xFFFF_FFFF)):
        got = _grads(q, k, v, do, p, seed, offset, causal)
        _compare(q, k, v, do, got, p, seed, offset, causal)


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal,p", [
    (1, 1, 1, 700, 128, False, 0.5),   # one query row
    (1, 2, 5, 1, 64, False, 0.5),      # one key
    (1, 1, 1, 1, 64, False, 0.3),
    (1, 1, 2, 2, 128, True, 0.5),
    (1, 2, 200, 333, 64, False, 0.99),  # t = 253: three bytes in 256 kept, s = 256 / 3
])
def test_parity_edge_shapes(B, H, Lq, Lk, D, causal, p):
    q, k, v, do = _inputs(B, H, Lq, Lk, D, seed=Lq * 7 + Lk)
    got = _grads(q, k, v, do, p, 99, 3, causal)
    _compare(q, k, v, do, got, p, 99, 3, causal)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_parity_sharp_logits(D, causal):
    q, k, v, do = _inputs(1, 2, 512, 512, D, seed=99, std=3.0)
    got = _grads(q, k, v, do, 0.3, 2024, 9, causal)
    _compare(q, k, v, do, got, 0.3, 2024, 9, causal)


@pytest.mark.parametrize("D,causal", [(64, False), (64, True), (128, False), (128, True)])
def test_p_zero_is_the_plain_backward(D, causal):
    q, k, v, do = _inputs(2, 2, 384, 384, D, seed=21)
    o, lse = fa.forward(q, k, v, causal=causal)
    plain = fa.backward(q, k, v, o, lse, do, causal=causal)
    drop = fa.backward_dropout(q, k, v, o, lse, do, 0.0, 77, 5, causal=causal)
    _check()
    for a, b in zip(plain, drop):
        assert torch.equal(a, b)
    # a drop probability that rounds to t = 0 keeps every weight too
    tiny = fa.backward_dropout(q, k, v, o, lse, do, 0.001, 77, 5, causal=causal)
    for a, b in zip(plain, tiny):
        assert torch.equal(a, b)


def _unit_rows(n, D, lo=0, hi=None):
    """Rows e_(i mod D) for i in [lo, hi), zero rows elsewhere: [1, 1, n, D] bf16."""
    hi = n if hi is None else hi
    x = torch.zeros(n, D, dtype=torch.bfloat16)
    i = torch.arange(lo, hi)
    x[i, i % D] = 1
    return x.view(1, 1, n, D)


@pytest.mark.parametrize("D,causal,L", [(64, False, 200), (64, True, 320), (128, False, 384), (128, True, 300)])
@pytest.mark.parametrize("p", [0.1, 0.5, 0.8])
def test_keep_bits_bit_exact(D, causal, L, p):
    seed, offset = 0x0123_4567_89AB_CDEF, 11
    t = od.drop_threshold(p)
    z = od.keep_mask(0, np.arange(L), L, t, seed, offset)
    visible = np.tril(np.ones((L, L), dtype=bool)) if causal else np.ones((L, L), dtype=bool)
    q = _unit_rows(L, D).cuda()
    k = q.clone()
    _, lse = fa.forward(q, k, q, causal=causal)
    zero_o = torch.zeros_like(q)
    g = torch.Generator().manual_seed(D + L)
    # random dO with magnitudes in [0.5, 1.5]: every weight gradient nonzero
    mag = torch.rand(1, 1, L, D, generator=g) + 0.5
    sign = torch.where(torch.rand(1, 1, L, D, generator=g) < 0.5, -1.0, 1.0)
    do_rand = (mag * sign).to(torch.bfloat16)
    nb = (L + D - 1) // D
    seen_v = np.zeros((L, L), dtype=bool)
    seen_q = np.zeros((L, L), dtype=bool)
    seen_k = np.zeros((L, L), dtype=bool)
    for blk in range(nb):
        lo, hi = blk * D, min(L, (blk + 1) * D)
        # dv[j, c] = s w z at (lo + c, j): the key-tile kernel's P path
        do_unit = _unit_rows(L, D, lo, hi).cuda()
        _, _, dv = fa.backward_dropout(q, k, q, zero_o, lse, do_unit, p, seed, offset, causal=causal)
        # dq[i, c] = scale dA[i, lo + c]: the query-tile kernel's bits
        v_blk = _unit_rows(L, D, lo, hi).cuda()
        dq, _, _ = fa.backward_dropout(q, k, v_blk, zero_o, lse, do_rand.cuda(), p, seed, offset,
                                       causal=causal)
        # dk[j, c] = scale dA[lo + c, j]: the key-tile kernel's dS path
        do_blk = do_rand.clone()
        do_blk[:, :, :lo] = 0
        do_blk[:, :, hi:] = 0
        _, dk, _ = fa.backward_dropout(q, k, q, zero_o, lse, do_blk.cuda(), p, seed, offset, causal=causal)
        _check()
        nz_v = to_f64(dv[0, 0].cpu())[:, :hi - lo].T != 0      # [query lo..hi, key]
        nz_q = to_f64(dq[0, 0].cpu())[:, :hi - lo] != 0        # [query, key lo..hi]
        nz_k = to_f64(dk[0, 0].cpu())[:, :hi - lo].T != 0      # [query lo..hi, key]
        rows, cols = slice(lo, hi), slice(lo, hi)
        vis_r, vis_c = visible[rows, :], visible[:, cols]
        assert np.array_equal(nz_v[vis_r], z[rows, :][vis_r]), ("dv", blk)
        assert not nz_v[~vis_r].any()
        assert np.array_equal(nz_q[vis_c], z[:, cols][vis_c]), ("dq", blk)
        assert not nz_q[~vis_c].any()
        assert np.array_equal(nz_k[vis_r], z[rows, :][vis_r]), ("dk", blk)
        assert not nz_k[~vis_r].any()
        seen_v[rows, :] = seen_k[rows, :] = True
        seen_q[:, cols] = True
    assert seen_v.all() and seen_q.all() and seen_k.all()


def test_seed_and_offset_select_different_bits():
    q, k, v, do = _inputs(1, 1, 256, 256, 128, seed=3)
    o, lse = fa.forward(q, k, v)
    runs = [fa.backward_dropout(q, k, v, o, lse, do, 0.5, s, off)
            for s, off in ((1, 0), (2, 0), (1, 1), (1 | (1 << 32), 0))]
    _check()
    for a in range(len(runs)):
        for b in range(a + 1, len(runs)):
            for x, y in zip(runs[a], runs[b]):
                assert not torch.equal(x, y)
    again = fa.backward_dropout(q, k, v, o, lse, do, 0.5, 1, 0)
    for x, y in zip(runs[0], again):
        assert torch.equal(x, y)


def test_invalid_drop_probability_is_rejected():
    q, k, v, do = _inputs(1, 1, 128, 128, 64, seed=4)
    o, lse = fa.forward(q, k, v)
    for p in (-0.1, 1.0, 0.999, float("nan"), float("inf")):
        with pytest.raises(fa.FlashAttentionError) as e:
            fa.backward_dropout(q, k, v, o, lse, do, p, 1, 0)
        assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_binding_rejects_bad_gradient_buffers():
    q, k, v, do = _inputs(1, 2, 128, 256, 64, seed=6)
    o, lse = fa.forward_dropout(q, k, v, 0.1, 1)
    for kw in (dict(dq=torch.empty_like(k)), dict(dk=torch.empty_like(q)),
               dict(dv=torch.empty(v.shape, dtype=torch.float32, device=v.device)),
               dict(dq=torch.empty_like(q).transpose(2, 3).contiguous().transpose(2, 3))):
        with pytest.raises(ValueError):
            fa.backward_dropout(q, k, v, o, lse, do, 0.1, 1, **kw)
        with pytest.raises(ValueError):
            fa.backward(q, k, v, o, lse, do, **kw)
    with pytest.raises(ValueError):
        fa.backward_dropout(q, k, v, o, lse[:, :, :64], do, 0.1, 1)


@pytest.mark.slow
def test_causal_l8k_d128_whole_heads():
    w = WORKLOADS["causal_l8k_d128"]
    dev = torch.device("cuda")
    q, k, v = make_inputs(w, dev)
    gen = torch.Generator(device=dev).manual_seed(11)
    do = torch.randn(q.shape, generator=gen, device=dev).to(torch.bfloat16)
    p, seed, offset = 0.1, 1234, 0
    dq, dk, dv = _grads(q, k, v, do, p, seed, offset, True)
    for bh in (0, 63):
        b, h = divmod(bh, w.H)
        refs = od.backward_dropout_head(to_f64(q[b, h].cpu()), to_f64(k[b, h].cpu()), to_f64(v[b, h].cpu()),
                                        to_f64(do[b, h].cpu()), w.scale, True, bh, p, seed, offset)
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            err = float(np.abs(to_f64(got[b, h].cpu()) - ref).max())
            mag = float(np.abs(ref).max())
            print(f"head {bh} {name}: max err {err:.3e}  max |ref| {mag:.3e}")
            assert err <= RTOL_GRAD * max(1.0, mag), (bh, name, err, mag)
        del refs
