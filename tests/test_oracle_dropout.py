"""Pins of the dropout oracle (oracle/dropout.py) and of its Philox generator
(oracle/philox.py), against things other than themselves:

* the generic Philox round, at 64-bit width, against numpy's library
  implementation (numpy.random.Philox, Philox-4x64-10; its first block is the
  one for counter + 1);
* the vectorised 32-bit path against the scalar generic routine;
* p = 0 reduces to plain attention (oracle.naive), and the log-sum-exp never
  depends on the dropout;
* the output is unbiased: its mean over many seeds approaches plain attention;
* the keep fraction and the byte distribution match the threshold;
* planted mistakes (no rescale, a wrong byte order, the sum taken over the
  dropped weights) fail these checks.
"""
import math

import numpy as np
import pytest

from oracle import dropout as od
from oracle import philox as ph
from oracle.naive import attention_rows


def test_philox_generic_round_matches_numpy_philox4x64():
    rng = np.random.default_rng(3)
    for _ in range(20):
        ctr = [int(x) for x in rng.integers(0, 2**63, size=4, dtype=np.int64)]
        ctr[0] = ctr[0] & ~1   # keep counter + 1 from carrying
        key = [int(x) for x in rng.integers(0, 2**63, size=2, dtype=np.int64)]
        bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
        lib = [int(x) for x in bg.random_raw(4)]
        nxt = list(ctr)
        nxt[0] += 1
        assert ph.philox4x64_10(nxt, key) == lib


def test_philox_zero_counter_reference_block():
    # the all-zero counter and key: numpy's block for counter 1 is the next one
    bg = np.random.Philox(counter=np.zeros(4, dtype=np.uint64), key=np.zeros(2, dtype=np.uint64))
    assert ph.philox4x64_10([1, 0, 0, 0], [0, 0]) == [int(x) for x in bg.random_raw(4)]


def test_philox4x32_vector_path_matches_scalar():
    rng = np.random.default_rng(4)
    c = rng.integers(0, 2**32, size=(4, 64), dtype=np.uint64)
    key = (0x12345678, 0x9ABCDEF0)
    vec = ph.philox4x32_10((c[0], c[1], c[2], c[3]), key)
    for n in range(64):
        assert [int(v[n]) for v in vec] == ph.philox(list(int(x) for x in c[:, n]), key, 32)


def test_philox4x32_is_not_the_64_bit_instance_truncated():
    # the two widths use different constants: the 32-bit outputs are not the
    # low halves of the 64-bit ones
    a = ph.philox([1, 2, 3, 4], [5, 6], 32)
    b = ph.philox4x64_10([1, 2, 3, 4], [5, 6])
    assert a != [x & 0xFFFFFFFF for x in b]


def _case(seed, R=48, L=80, D=16):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((R, D)), rng.standard_normal((L, D)), rng.standard_normal((L, D))


@pytest.mark.parametrize("causal", [False, True])
def test_p_zero_is_plain_attention(causal):
    q, k, v = _case(1)
    rows = np.arange(q.shape[0]) + (32 if causal else 0)
    o, lse, z = od.attention_dropout_rows(q, k, v, 0.25, causal, rows, 3, 0.0, 99, 0)
    o0, lse0 = attention_rows(q, k, v, 0.25, causal=causal, row_index=rows)
    assert z.all()
    np.testing.assert_allclose(o, o0, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(lse, lse0)


def test_lse_does_not_depend_on_dropout():
    q, k, v = _case(2)
    rows = np.arange(q.shape[0])
    _, lse0 = attention_rows(q, k, v, 0.3, row_index=rows)
    for p, seed in ((0.1, 1), (0.5, 2), (0.9, 3)):
        _, lse, z = od.attention_dropout_rows(q, k, v, 0.3, False, rows, 0, p, seed, 7)
        assert not z.all()
        np.testing.assert_array_equal(lse, lse0)


def test_threshold_quantisation():
    assert od.drop_threshold(0.0) == 0
    assert od.drop_threshold(0.1) == 26          # 25.6 -> 26
    assert od.drop_threshold(0.5) == 128
    assert od.drop_threshold(0.998) == 255       # 255.49 -> 255
    with pytest.raises(ValueError):
        od.drop_threshold(0.999)                 # 255.74 -> 256
    with pytest.raises(ValueError):
        od.drop_threshold(-0.1)
    with pytest.raises(ValueError):
        od.drop_threshold(1.0)


def test_keep_fraction_and_byte_uniformity():
    t = od.drop_threshold(0.3)
    z = od.keep_mask(5, np.arange(256), 4096, t, seed=2024, offset=3)
    n = z.size
    frac = z.mean()
    keep = (256 - t) / 256
    assert abs(frac - keep) < 5 * math.sqrt(keep * (1 - keep) / n)
    # the bytes themselves: chi-square over 256 bins
    rows = np.arange(64, dtype=np.uint64).reshape(-1, 1)
    g = np.arange(64, dtype=np.uint64).reshape(1, -1)
    x = ph.philox4x32_10((g, rows, np.uint64(1), np.uint64(0)), (11, 12))
    b = np.stack(x, -1).view(np.uint8).ravel()
    cnt = np.bincount(b, minlength=256)
    e = b.size / 256
    chi2 = ((cnt - e) ** 2 / e).sum()
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)


def test_mask_depends_on_every_counter_field():
    t = od.drop_threshold(0.5)
    base = od.keep_mask(1, np.arange(16), 64, t, seed=5, offset=0)
    for other in (od.keep_mask(2, np.arange(16), 64, t, seed=5, offset=0),          # head
                  od.keep_mask(1, np.arange(16, 32), 64, t, seed=5, offset=0),     # rows
                  od.keep_mask(1, np.arange(16), 64, t, seed=6, offset=0),         # seed, low word
                  od.keep_mask(1, np.arange(16), 64, t, seed=5 + (1 << 32), offset=0),  # seed, high word
                  od.keep_mask(1, np.arange(16), 64, t, seed=5, offset=1)):        # offset
        assert (base != other).mean() > 0.3
    # key groups of 16: columns 0-15 and 16-31 come from different calls
    assert (base[:, :16] != base[:, 16:32]).mean() > 0.3


def test_byte_layout_within_a_call():
    # key j of row i takes byte j % 4 of word (j // 4) % 4 of call (j // 16, i, bh, offset)
    t = 128
    z = od.keep_mask(7, [3], 32, t, seed=0xABCDEF0123, offset=9)
    for grp in range(2):
        words = ph.philox([grp, 3, 7, 9], [0xABCDEF0123 & 0xFFFFFFFF, 0xABCDEF0123 >> 32], 32)
        for j in range(16):
            byte = (words[j // 4] >> (8 * (j % 4))) & 0xFF
            assert z[0, 16 * grp + j] == (byte >= t)


def _draws(fn, n, q, k, v, rows):
    return np.stack([fn(q, k, v, 0.5, False, rows, 0, 0.4, s, 0)[0] for s in range(n)])


def _within_6_sigma(draws, target):
    """Every entry's mean over the draws within 6 standard errors (from the
    draws' own spread) of the target."""
    n = draws.shape[0]
    se = draws.std(axis=0, ddof=1) / math.sqrt(n)
    return bool((np.abs(draws.mean(axis=0) - target) <= 6 * se + 1e-12).all())


def test_output_is_unbiased():
    q, k, v = _case(3, R=8, L=24, D=4)
    rows = np.arange(8)
    o0, _ = attention_rows(q, k, v, 0.5, row_index=rows)
    assert _within_6_sigma(_draws(od.attention_dropout_rows, 800, q, k, v, rows), o0)


def test_planted_mistakes_fail():
    q, k, v = _case(3, R=8, L=24, D=4)
    rows = np.arange(8)
    o0, lse0 = attention_rows(q, k, v, 0.5, row_index=rows)

    def no_rescale(q, k, v, scale, causal, rows, bh, p, seed, off):
        o, lse, z = od.attention_dropout_rows(q, k, v, scale, causal, rows, bh, p, seed, off)
        return o * (256 - od.drop_threshold(p)) / 256, lse, z

    def renormalised(q, k, v, scale, causal, rows, bh, p, seed, off):
        # the sum over the kept weights instead of all of them
        _, _, w = attention_rows(q, k, v, scale, row_index=rows, return_weights=True)
        z = od.keep_mask(bh, rows, k.shape[0], od.drop_threshold(p), seed, off)
        wz = w * z
        s = np.maximum(wz.sum(1, keepdims=True), 1e-300)
        return (wz / s) @ v, None, z

    assert not _within_6_sigma(_draws(no_rescale, 800, q, k, v, rows), o0)
    assert not _within_6_sigma(_draws(renormalised, 800, q, k, v, rows), o0)

    # a wrong byte order (big-endian bytes) changes the mask
    t = 128
    z = od.keep_mask(0, np.arange(8), 64, t, seed=1, offset=0)
    x = ph.philox4x32_10((np.arange(4, dtype=np.uint64).reshape(1, -1), np.arange(8, dtype=np.uint64).reshape(-1, 1),
                          np.uint64(0), np.uint64(0)), (1, 0))
    be = np.stack(x, -1).astype(">u4").view(np.uint8).reshape(8, -1)[:, :64] >= t
    assert (be != z).mean() > 0.3


# ---------------------------------------------------------------- backward

def _bw_case(seed, Lq=6, Lk=9, D=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Lq, D)), rng.standard_normal((Lk, D)),
            rng.standard_normal((Lk, D)), rng.standard_normal((Lq, D)))


def _dropout_forward(q, k, v, scale, causal, bh, p, seed, offset):
    o, _, _ = od.attention_dropout_rows(q, k, v, scale, causal, np.arange(q.shape[0]), bh, p, seed, offset)
    return o


def _fd_check(grads, q, k, v, do, scale, causal, bh, p, seed, offset, rng_seed):
    """Central differences of <dO, O> along random directions, the keep mask
    fixed by the seed; returns the worst relative mismatch."""
    f = lambda q_, k_, v_: float((do * _dropout_forward(q_, k_, v_, scale, causal, bh, p, seed, offset)).sum())
    rng = np.random.default_rng(rng_seed)
    h = 1e-5
    worst = 0.0
    for which, g in zip(("q", "k", "v"), grads):
        for _ in range(3):
            u = rng.standard_normal(g.shape)
            ap = {"q": q, "k": k, "v": v}
            am = dict(ap)
            ap[which] = ap[which] + h * u
            am[which] = am[which] - h * u
            fd = (f(ap["q"], ap["k"], ap["v"]) - f(am["q"], am["k"], am["v"])) / (2 * h)
            worst = max(worst, abs(fd - float((g * u).sum())) / max(1.0, abs(fd)))
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.3, 0.75])
def test_backward_finite_differences(causal, p):
    q, k, v, do = _bw_case(11)
    if causal:
        k, v = k[:6], v[:6]
    scale, bh, seed, offset = 0.7, 5, 0x0123_4567_89AB_CDEF, 9
    grads = od.backward_dropout_head(q, k, v, do, scale, causal, bh, p, seed, offset)
    assert _fd_check(grads, q, k, v, do, scale, causal, bh, p, seed, offset, 12) <= 1e-7
    # the mask matters: at this p some weights are dropped
    z = od.keep_mask(bh, np.arange(6), k.shape[0], od.drop_threshold(p), seed, offset)
    assert not z.all()


def test_backward_p_zero_is_the_plain_backward():
    from oracle.backward import backward_head
    q, k, v, do = _bw_case(13)
    for causal in (False, True):
        kk, vv = (k[:6], v[:6]) if causal else (k, v)
        a = od.backward_dropout_head(q, kk, vv, do, 0.4, causal, 2, 0.0, 1, 0)
        b = backward_head(q, kk, vv, do, 0.4, causal)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)


def test_backward_row_term_equals_rowsum_do_times_o():
    # rowsum(w * dW) (the oracle's form) = rowsum(dO * O) with O the dropout
    # forward's output (the form the kernels compute once per row)
    q, k, v, do = _bw_case(14)
    scale, bh, p, seed, offset = 0.5, 1, 0.4, 77, 3
    t = od.drop_threshold(p)
    s = 256.0 / (256.0 - t)
    _, _, w = attention_rows(q, k, v, scale, causal=False, row_index=np.arange(6), return_weights=True)
    z = od.keep_mask(bh, np.arange(6), k.shape[0], t, seed, offset)
    dw = s * z * (do @ v.T)
    o = _dropout_forward(q, k, v, scale, False, bh, p, seed, offset)
    np.testing.assert_allclose((w * dw).sum(1), (do * o).sum(1), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", ["dV without the mask", "dW without the scale", "row term of undropped weights",
                                  "mask on dQ only"])
def test_backward_planted_mistakes_fail_finite_differences(kind):
    q, k, v, do = _bw_case(15)
    scale, bh, p, seed, offset = 0.6, 4, 0.5, 2024, 0

    def mutant():
        t = od.drop_threshold(p)
        s = 256.0 / (256.0 - t)
        _, _, w = attention_rows(q, k, v, scale, causal=False, row_index=np.arange(6), return_weights=True)
        z = od.keep_mask(bh, np.arange(6), k.shape[0], t, seed, offset).astype(float)
        dv = s * ((w * z).T @ do) if kind != "dV without the mask" else s * (w.T @ do)
        dwz = do @ v.T
        dw = s * z * dwz if kind != "dW without the scale" else z * dwz
        if kind == "row term of undropped weights":
            da = w * (dw - (w * dwz).sum(1, keepdims=True))
        else:
            da = w * (dw - (w * dw).sum(1, keepdims=True))
        dq = scale * (da @ k)
        if kind == "mask on dQ only":
            da2 = w * (dwz - (w * dwz).sum(1, keepdims=True))
            return dq, scale * (da2.T @ q), dv
        return dq, scale * (da.T @ q), dv

    assert _fd_check(mutant(), q, k, v, do, scale, False, bh, p, seed, offset, 16) > 1e-3
    # and the oracle itself passes the same check
    good = od.backward_dropout_head(q, k, v, do, scale, False, bh, p, seed, offset)
    assert _fd_check(good, q, k, v, do, scale, False, bh, p, seed, offset, 16) <= 1e-7
