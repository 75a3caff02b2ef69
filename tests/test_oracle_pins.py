"""Pins for the fp64 oracle, independent of the oracle itself.

Each check ties the oracle to something the pages or plain mathematics fix:
hand-worked values from the pages' examples (tests/golden), the guide's
rescale identity and chunk recurrence, closed forms and invariants, a
pure-Python brute force on tiny inputs, and scipy's logsumexp.  A last test
plants plausible mistakes in a copy of the oracle and checks that at least one
pin catches every one of them.
"""
import inspect
import json
import math
import os
import textwrap

import numpy as np
import pytest

from oracle import naive as oracle_mod
from oracle.naive import attention, attention_head, attention_rows
from oracle.recurrence import (online_attention_row, online_softmax_stats,
                               rescale_identity_sides)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Pins written against a rows-function with the signature of attention_rows,
# so the mutation test can run them on planted mistakes.
# --------------------------------------------------------------------------

def pin_single_query(fn):
    g = _load("single_query_d2_l3.json")
    o, lse, w = fn(np.array([g["q"]]), np.array(g["k"]), np.array(g["v"]),
                   g["scale"], return_weights=True)
    assert np.allclose(w[0], g["weights"], rtol=1e-14, atol=1e-15)
    assert np.allclose(o[0], g["O"], rtol=1e-14, atol=1e-15)
    assert abs(lse[0] - g["LSE"]) < 1e-14
    # the same values from the closed forms, written independently
    e = math.e
    z = 1 + e + e * e
    assert np.allclose(o[0], [(1 + e * e) / z, (e + e * e) / z], rtol=1e-14)
    assert abs(lse[0] - math.log(z)) < 1e-14


def pin_scaled_single_query(fn):
    # scale 0.5 on the hand case: a = [0, 0.5, 1]
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.0, 0.0], [1.0, 0.0], [2.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    o, lse = fn(q, k, v, 0.5)
    e = [1.0, math.exp(0.5), math.exp(1.0)]
    z = sum(e)
    assert np.allclose(o[0], [(e[0] + e[2]) / z, (e[1] + e[2]) / z], rtol=1e-14)
    assert abs(lse[0] - math.log(z)) < 1e-14


def pin_worked_example(fn):
    g = _load("softmax_blocks_1234.json")
    x = g["vector"]
    q = np.array([[1.0, 0.0, 0.0, 0.0]])
    k = np.array([[xi, 0.0, 0.0, 0.0] for xi in x])
    v = np.eye(4)
    o, lse, w = fn(q, k, v, 1.0, return_weights=True)
    assert np.allclose(w[0], g["softmax"], rtol=1e-14)
    assert np.allclose(o[0], g["softmax"], rtol=1e-14)   # one-hot values read the weights out
    assert abs(lse[0] - (g["merged"]["m"] + math.log(g["merged"]["l"]))) < 1e-14


def pin_brute_force(fn):
    # pure-Python loops over the definition, asymmetric tiny shapes
    rng = np.random.default_rng(11)
    Lq, Lk, D, scale = 3, 5, 4, 0.7
    q = rng.standard_normal((Lq, D))
    k = rng.standard_normal((Lk, D))
    v = rng.standard_normal((Lk, D))
    for causal in (False, True):
        o, lse = fn(q, k, v, scale, causal=causal, row_index=np.arange(Lq))
        for i in range(Lq):
            keys = [j for j in range(Lk) if (not causal or j <= i)]
            a = [scale * sum(q[i][d] * k[j][d] for d in range(D)) for j in keys]
            amax = max(a)
            e = [math.exp(x - amax) for x in a]
            s = sum(e)
            ref = [sum(e[n] / s * v[j][d] for n, j in enumerate(keys)) for d in range(D)]
            assert np.allclose(o[i], ref, rtol=1e-13, atol=1e-14)
            assert abs(lse[i] - (amax + math.log(s))) < 1e-13


def pin_causal_edges(fn):
    rng = np.random.default_rng(5)
    L, D, scale = 7, 3, 0.9
    q, k, v = (rng.standard_normal((L, D)) for _ in range(3))
    o, lse = fn(q, k, v, scale, causal=True, row_index=np.arange(L))
    # row 0 sees only key 0
    assert np.allclose(o[0], v[0], rtol=1e-15, atol=1e-15)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-14
    # the last row sees every key: equal to the non-causal result
    o_nc, lse_nc = fn(q[-1:], k, v, scale)
    assert np.allclose(o[-1], o_nc[0], rtol=1e-14, atol=1e-15)
    assert abs(lse[-1] - lse_nc[0]) < 1e-14


def pin_large_logits(fn):
    # scores c + x_j with c = 1000: a softmax without the max subtraction
    # overflows; weights must equal softmax(x) and LSE = c + logsumexp(x)
    c = 1000.0
    x = np.array([0.3, -1.2, 2.0, 0.0])
    q = np.array([[c, 1.0]])
    k = np.stack([np.ones_like(x), x], axis=1)
    v = np.eye(4)[:, :4]
    v = np.concatenate([v, np.zeros((4, 0))], axis=1)
    o, lse, w = fn(q, k, v, 1.0, return_weights=True)
    ex = np.exp(x - x.max())
    assert np.all(np.isfinite(o)) and np.isfinite(lse[0])
    assert np.allclose(w[0], ex / ex.sum(), rtol=1e-12)
    assert abs(lse[0] - (c + x.max() + math.log(ex.sum()))) < 1e-10


PINS = [pin_single_query, pin_scaled_single_query, pin_worked_example,
        pin_brute_force, pin_causal_edges, pin_large_logits]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(attention_rows)


# --------------------------------------------------------------------------
# The guide's identities and recurrence
# --------------------------------------------------------------------------

def test_worked_example_block_statistics():
    """The (d, s) recurrence on [1,2,3,4] in blocks of 2 reproduces the
    page's two block statistics and the merged denominator."""
    g = _load("softmax_blocks_1234.json")
    stats = online_softmax_stats(g["vector"], 2)
    (d1, s1), (d2, s2) = stats
    assert d1 == g["block1"]["m"] and abs(s1 - g["block1"]["l"]) < 1e-15
    assert d2 == g["merged"]["m"] and abs(s2 - g["merged"]["l"]) < 1e-15
    # block 2 on its own
    (d2b, s2b), = online_softmax_stats(g["blocks"][1], 2)
    assert d2b == g["block2"]["m"] and abs(s2b - g["block2"]["l"]) < 1e-15
    assert abs(s1 * math.exp(d1 - d2b) + s2b - g["merged"]["l"]) < 1e-15


@pytest.mark.parametrize("seed", range(20))
def test_rescale_identity_per_tile(seed):
    """s1 * exp(d1 - d2) == sum exp(a_i - d2) for a chunk with max d1 and any
    later reference d2 (the guide's one formula)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(rng.integers(1, 200)) * rng.uniform(0.1, 20)
    d1 = a.max()
    for d2 in (d1, d1 + rng.uniform(0, 10), d1 - rng.uniform(0, 3)):
        lhs, rhs = rescale_identity_sides(a, d1, d2)
        assert abs(lhs - rhs) <= 1e-13 * abs(rhs)


def test_recurrence_ends_at_amax_and_full_denominator():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(50) * 4
    full = np.exp(a - a.max()).sum()
    for chunk in range(1, 51):
        d, s = online_softmax_stats(a, chunk)[-1]
        assert d == a.max()
        assert abs(s - full) <= 1e-13 * full


@pytest.mark.parametrize("causal", [False, True])
def test_recurrence_equals_two_pass_every_chunk(causal):
    """The guide's one-pass O recurrence equals the oracle's two-pass result
    for every chunk size 1..L on tiny inputs."""
    rng = np.random.default_rng(7 + causal)
    L, D, scale = 19, 6, 0.45
    q, k, v = (rng.standard_normal((L, D)) * 2 for _ in range(3))
    o_ref, lse_ref = attention_head(q, k, v, scale, causal=causal)
    for chunk in range(1, L + 1):
        for i in range(L):
            o, d, s = online_attention_row(q[i], k, v, scale, chunk,
                                           n_visible=(i + 1) if causal else None)
            assert np.allclose(o, o_ref[i], rtol=1e-12, atol=1e-13)
            assert abs(d + math.log(s) - lse_ref[i]) <= 1e-12 * max(1.0, abs(lse_ref[i]))


# --------------------------------------------------------------------------
# Invariants and special cases
# --------------------------------------------------------------------------

def test_weights_rows_sum_to_one():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((16, 8)) * 3 for _ in range(3))
    for causal in (False, True):
        _, _, w = attention_rows(q, k, v, 0.5, causal=causal, row_index=np.arange(16),
                                 return_weights=True)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-14)
        if causal:
            assert np.all(np.triu(w, 1) == 0.0)


def test_constant_v_returns_v():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((9, 5)), rng.standard_normal((11, 5))
    row = rng.standard_normal(5)
    v = np.tile(row, (11, 1))
    o, _ = attention_rows(q, k, v, 1.3)
    assert np.allclose(o, np.tile(row, (9, 1)), rtol=1e-14, atol=1e-15)


def test_scale_zero_gives_mean_and_log_length():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((4, 6)), rng.standard_normal((10, 6)), rng.standard_normal((10, 6))
    o, lse = attention_rows(q, k, v, 0.0)
    assert np.allclose(o, np.tile(v.mean(axis=0), (4, 1)), rtol=1e-14, atol=1e-15)
    assert np.allclose(lse, math.log(10), rtol=1e-15)


def test_single_key():
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal((3, 4)), rng.standard_normal((1, 4)), rng.standard_normal((1, 4))
    o, lse = attention_rows(q, k, v, 0.8)
    assert np.allclose(o, np.tile(v[0], (3, 1)), rtol=1e-15)
    assert np.allclose(lse, 0.8 * (q @ k[0]), rtol=1e-14)


def test_joint_key_value_permutation_invariance():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((5, 7)), rng.standard_normal((13, 7)), rng.standard_normal((13, 7))
    perm = rng.permutation(13)
    o1, l1 = attention_rows(q, k, v, 0.6)
    o2, l2 = attention_rows(q, k[perm], v[perm], 0.6)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-14) and np.allclose(l1, l2, rtol=1e-14)


def test_against_scipy_logsumexp():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(9)
    B, H, L, D, scale = 2, 3, 17, 8, 0.35
    q, k, v = (rng.standard_normal((B, H, L, D)) for _ in range(3))
    o, lse = attention(q, k, v, scale)
    for b in range(B):
        for h in range(H):
            s = scale * np.einsum("id,jd->ij", q[b, h], k[b, h])
            ref_lse = special.logsumexp(s, axis=1)
            ref_o = special.softmax(s, axis=1) @ v[b, h]
            assert np.allclose(lse[b, h], ref_lse, rtol=1e-14)
            assert np.allclose(o[b, h], ref_o, rtol=1e-13, atol=1e-14)


def test_bf16_widening_is_exact():
    torch = pytest.importorskip("torch")
    x = torch.randn(1000).to(torch.bfloat16)
    y = oracle_mod.to_f64(x)
    assert y.dtype == np.float64
    assert np.array_equal(y.astype(np.float32), x.float().numpy())


# --------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "mask_direction": ("np.where(j <= i, a, -np.inf)", "np.where(j >= i, a, -np.inf)"),
    "mask_strict": ("np.where(j <= i, a, -np.inf)", "np.where(j < i, a, -np.inf)"),
    "dropped_scale": ("a = float(scale) * (q_rows @ k.T)", "a = (q_rows @ k.T)"),
    "min_not_max": ("amax = a.max(axis=1)", "amax = a.min(axis=1)"),
    "no_max_subtraction": ("e = np.exp(a - amax_safe[:, None])", "e = np.exp(a)"),
    "exp2_not_exp": ("e = np.exp(a - amax_safe[:, None])", "e = np.exp2(a - amax_safe[:, None])"),
    "no_normalisation": ("w = e / s_safe[:, None]", "w = e"),
    "lse_log2": ("amax_safe + np.log(s_safe)", "amax_safe + np.log2(s_safe)"),
    "lse_missing_max": ("amax_safe + np.log(s_safe)", "np.log(s_safe)"),
    "weights_times_keys": ("o = w @ v", "o = w @ k"),
}


def _mutant(old, new):
    src = textwrap.dedent(inspect.getsource(attention_rows))
    assert old in src, old
    ns = {"np": np}
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["attention_rows"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    fn = _mutant(*MUTANTS[name])
    caught = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(fn)
        except (AssertionError, ValueError, FloatingPointError):
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name}"
