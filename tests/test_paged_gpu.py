"""GPU parity of single-query attention against a paged cache
(fa_fwd_decode_paged through the C ABI) with the fp64 oracle oracle.paged:
every row at small sizes (ragged lengths, lengths of one position, a page,
a page and one, the table's capacity, empty sequences, page sizes 1..128,
pages in random order), sampled heads at 128K cached positions, and the
bounds check on page ids."""
import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import PAGED_WORKLOADS, PagedWorkload, make_paged_inputs
from oracle.paged import decode_paged as oracle_paged
from parity_util import ATOL_LSE, ATOL_O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _check(q, kc, vc, bt, lens, scale, heads=None):
    o, lse = fa.decode_paged(q, kc, vc, bt, lens, scale=scale)
    st, site = fa.last_device_error()
    assert st == fa.FA_OK, (st, site)
    if heads is None:
        ro, rl = oracle_paged(q.cpu(), kc.cpu(), vc.cpu(), bt.cpu(), lens.cpu(), scale)
        go = o.float().cpu().numpy().astype(np.float64)
        gl = lse.cpu().numpy().astype(np.float64)
    else:
        # only the selected (b, h) pairs: gather those sequences on the host
        bs = sorted({b for b, _ in heads})
        sel = torch.tensor(bs)
        ro_all, rl_all = oracle_paged(q[sel].cpu(), kc.cpu(), vc.cpu(), bt[sel].cpu(), lens[sel].cpu(), scale)
        idx = {b: i for i, b in enumerate(bs)}
        ro = np.stack([ro_all[idx[b], h] for b, h in heads])
        rl = np.array([rl_all[idx[b], h] for b, h in heads])
        go = np.stack([o[b, h].float().cpu().numpy() for b, h in heads]).astype(np.float64)
        gl = np.array([lse[b, h].item() for b, h in heads], dtype=np.float64)
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(gl), empty)
    assert np.all(go[empty] == 0)
    d_o = np.abs(go - ro).max() if go.size else 0.0
    d_l = np.abs(gl[~empty] - rl[~empty]).max() if (~empty).any() else 0.0
    assert d_o <= ATOL_O, f"max |dO| = {d_o:.3e}"
    assert d_l <= ATOL_LSE, f"max |dLSE| = {d_l:.3e}"
    return o, lse


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("page_size", [1, 16, 128])
def test_ragged_lengths(D, page_size):
    lengths = (1, page_size, page_size + 1, 3 * page_size - 1, min(700, 64 * page_size) - 1,
               64 * page_size)
    w = PagedWorkload("t", len(lengths), 4, D, page_size, 64 * page_size, 11, lengths=lengths)
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    _check(q, kc, vc, bt, lens, w.scale)


def test_drawn_lengths_and_custom_scale():
    w = PagedWorkload("t", 6, 8, 128, 32, 5000, 12)
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    _check(q, kc, vc, bt, lens, 0.37)


def test_empty_sequence_and_clamped_length():
    w = PagedWorkload("t", 3, 2, 64, 16, 64, 13, lengths=(5, 0, 64))
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    o, lse = _check(q, kc, vc, bt, lens, w.scale)
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(lse[1]))
    # a length above the table's capacity reads like the capacity
    lens2 = lens.clone()
    lens2[2] = 10 ** 6
    o2, lse2 = fa.decode_paged(q, kc, vc, bt, lens2, scale=w.scale)
    assert torch.equal(o2, o) and torch.equal(lse2, lse)


def test_page_id_out_of_range_is_recorded_not_read():
    w = PagedWorkload("t", 2, 2, 128, 16, 64, 14, lengths=(40, 40))
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    good_o, good_lse = _check(q, kc, vc, bt, lens, w.scale)
    bad = bt.clone()
    bad[1, 1] = kc.shape[0] + 1000          # read: positions 16..31 of sequence 1
    fa.last_device_error()                  # clear
    o, lse = fa.decode_paged(q, kc, vc, bad, lens, scale=w.scale)
    st, site = fa.last_device_error()
    assert st == fa.FA_ERR_INVALID_ARG and site == 11
    assert torch.equal(o[0], good_o[0]) and torch.equal(lse[0], good_lse[0])
    assert torch.isfinite(lse[1]).all()


def test_decode_paged_128k_sampled_heads():
    w = PAGED_WORKLOADS["decode_paged_128k_d128"]
    q, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
    g = torch.Generator().manual_seed(77)
    pick = torch.randperm(w.B * w.H, generator=g)[:24].tolist()
    heads = [(i // w.H, i % w.H) for i in pick]
    o, lse = _check(q, kc, vc, bt, lens, w.scale, heads=heads)
    assert torch.isfinite(lse).all()
    del q, kc, vc
    torch.cuda.empty_cache()
