"""Pins of the paged-cache oracle (oracle.paged) against facts that do not
come from it: an independent re-gathering with plain Python loops and
scipy's logsumexp, invariance under renumbering the physical pages, the
closed forms of one- and zero-position sequences, length clamping, and a
check that planted indexing mistakes in a copy of the gather are caught."""
import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import paged
from oracle.paged import decode_paged


def _case(seed, B=3, H=2, D=8, page_size=4, max_pages=5, num_pages=20):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, D))
    kc = rng.standard_normal((num_pages, page_size, H, D))
    vc = rng.standard_normal((num_pages, page_size, H, D))
    bt = np.stack([rng.permutation(num_pages)[:max_pages] for _ in range(B)])
    lens = np.array([max_pages * page_size, 1 + page_size, 7][:B])
    return q, kc, vc, bt, lens


def _reference(q, kc, vc, bt, lens, scale):
    """Independent: walk the pages one by one, append rows, then softmax."""
    B, H, D = q.shape
    ps = kc.shape[1]
    o = np.zeros((B, H, D))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(min(max(lens[b], 0), bt.shape[1] * ps))
        for h in range(H):
            keys, vals = [], []
            for pos in range(L):
                page = bt[b][pos // ps]
                keys.append(kc[page, pos % ps, h])
                vals.append(vc[page, pos % ps, h])
            if not keys:
                continue
            a = scale * np.array(keys) @ q[b, h]
            lse[b, h] = logsumexp(a)
            o[b, h] = np.exp(a - lse[b, h]) @ np.array(vals)
    return o, lse


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_independent_gather(seed):
    q, kc, vc, bt, lens = _case(seed)
    o, lse = decode_paged(q, kc, vc, bt, lens, 0.35)
    ro, rl = _reference(q, kc, vc, bt, lens, 0.35)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_renumbering_pages_changes_nothing():
    q, kc, vc, bt, lens = _case(5)
    perm = np.random.default_rng(9).permutation(kc.shape[0])   # new page id of old page i
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    o1, l1 = decode_paged(q, kc, vc, bt, lens, 0.5)
    o2, l2 = decode_paged(q, kc2, vc2, perm[bt], lens, 0.5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_one_position_and_empty_sequences():
    q, kc, vc, bt, _ = _case(3)
    lens = np.array([1, 0, 1])
    o, lse = decode_paged(q, kc, vc, bt, lens, 0.7)
    for b in (0, 2):
        page = bt[b, 0]
        np.testing.assert_allclose(o[b], vc[page, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[b], 0.7 * np.einsum("hd,hd->h", q[b], kc[page, 0]),
                                   rtol=0, atol=1e-14)
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))


def test_lengths_are_clamped_to_the_table():
    q, kc, vc, bt, _ = _case(4)
    cap = bt.shape[1] * kc.shape[1]
    o1, l1 = decode_paged(q, kc, vc, bt, np.array([cap, -3, cap]), 0.3)
    o2, l2 = decode_paged(q, kc, vc, bt, np.array([cap + 50, 0, 10 ** 9]), 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


_GATHER = paged.gather_sequence

MUTANTS = {
    "row off by one": lambda kc, vc, t, L, ps: (kc[np.asarray(t)[np.arange(L) // ps], (np.arange(L) + 1) % ps],
                                               vc[np.asarray(t)[np.arange(L) // ps], (np.arange(L) + 1) % ps]),
    "page index not divided": lambda kc, vc, t, L, ps: (kc[np.asarray(t)[np.arange(L) % len(t)], np.arange(L) % ps],
                                                       vc[np.asarray(t)[np.arange(L) % len(t)], np.arange(L) % ps]),
    "physical page = logical page": lambda kc, vc, t, L, ps: (kc[np.arange(L) // ps, np.arange(L) % ps],
                                                             vc[np.arange(L) // ps, np.arange(L) % ps]),
    "keys and values swapped": lambda kc, vc, t, L, ps: _GATHER(vc, kc, t, L, ps),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_gather_mistakes_are_caught(name, monkeypatch):
    q, kc, vc, bt, lens = _case(7)
    ro, rl = _reference(q, kc, vc, bt, lens, 0.4)
    monkeypatch.setattr(paged, "gather_sequence", MUTANTS[name])
    o, lse = paged.decode_paged(q, kc, vc, bt, lens, 0.4)
    assert not (np.allclose(o, ro, atol=1e-9) and np.allclose(lse, rl, atol=1e-9))
