"""Pins of the backward oracle against facts that do not come from it:
central finite differences of <dO, O> along random directions (O from the
forward oracle), torch.autograd in fp64, the closed form for values that do
not depend on the key (dQ = dK = 0), and planted mistakes in a copy of the
formulas that these pins catch."""
import numpy as np
import pytest

from oracle import backward as bw
from oracle.naive import attention_rows


def _forward(q, k, v, scale, causal):
    o, _ = attention_rows(q, k, v, scale, causal=causal, row_index=np.arange(q.shape[0]))
    return o


def _case(seed, Lq=6, Lk=6, D=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Lq, D)), rng.standard_normal((Lk, D)),
            rng.standard_normal((Lk, D)), rng.standard_normal((Lq, D)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_finite_differences(seed, causal):
    q, k, v, do = _case(seed)
    scale = 0.6
    dq, dk, dv = bw.backward_head(q, k, v, do, scale, causal)
    f = lambda q_, k_, v_: float((do * _forward(q_, k_, v_, scale, causal)).sum())
    rng = np.random.default_rng(seed + 10)
    h = 1e-5
    for which, g in (("q", dq), ("k", dk), ("v", dv)):
        for _ in range(3):
            u = rng.standard_normal(g.shape)
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[which] = args_p[which] + h * u
            args_m[which] = args_m[which] - h * u
            fd = (f(args_p["q"], args_p["k"], args_p["v"]) - f(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            assert abs(fd - float((g * u).sum())) <= 1e-7 * max(1.0, abs(fd)), which


def test_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    q, k, v, do = _case(3, Lq=5, Lk=7, D=3)
    scale = 0.8
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.softmax(scale * tq @ tk.T, dim=-1) @ tv
    o.backward(torch.tensor(do))
    dq, dk, dv = bw.backward_head(q, k, v, do, scale)
    for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-12, atol=1e-13)


def test_values_equal_for_every_key_give_zero_dq_dk():
    q, k, _, do = _case(4)
    v = np.tile(np.random.default_rng(5).standard_normal((1, 4)), (6, 1))
    dq, dk, dv = bw.backward_head(q, k, v, do, 0.5)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-13)   # sum of weights is 1


_ORIGINAL = bw.backward_head


def _mutant(kind):
    def f(q, k, v, do, scale, causal=False):
        a = scale * (q @ k.T)
        if causal:
            a = np.where(np.arange(k.shape[0])[None, :] <= np.arange(q.shape[0])[:, None], a, -np.inf)
        p = np.exp(a - a.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        dp = do @ v.T
        da = p * (dp - (p * dp).sum(1, keepdims=True))
        if kind == "no D term":
            da = p * dp
        if kind == "dS transposed":
            return scale * (da.T @ k if da.shape[0] == da.shape[1] else da @ k), scale * (da @ q), p.T @ do
        if kind == "scale missing":
            return da @ k, da.T @ q, p.T @ do
        if kind == "dV from P":
            return scale * (da @ k), scale * (da.T @ q), p @ do
        return scale * (da @ k), scale * (da.T @ q), p.T @ do
    return f


@pytest.mark.parametrize("kind", ["no D term", "dS transposed", "scale missing", "dV from P"])
def test_planted_mistakes_fail_the_finite_differences(kind):
    q, k, v, do = _case(6)
    scale = 0.6
    dq, dk, dv = _mutant(kind)(q, k, v, do, scale)
    f = lambda q_, k_, v_: float((do * _forward(q_, k_, v_, scale, False)).sum())
    rng = np.random.default_rng(7)
    h = 1e-5
    bad = False
    for which, g in (("q", dq), ("k", dk), ("v", dv)):
        u = rng.standard_normal(g.shape)
        a = {"q": q, "k": k, "v": v}
        b = dict(a)
        a[which] = a[which] + h * u
        b[which] = b[which] - h * u
        fd = (f(a["q"], a["k"], a["v"]) - f(b["q"], b["k"], b["v"])) / (2 * h)
        bad |= abs(fd - float((g * u).sum())) > 1e-6 * max(1.0, abs(fd))
    assert bad
