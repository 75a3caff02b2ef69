"""Pins of the row-softmax oracle against facts that do not come from it:
scipy's softmax and logsumexp, rows summing to one, invariance under adding
a constant to a row, closed forms (a constant row is uniform; two values give
the logistic function), the empty-row convention, and the two-read recurrence
of the guide reaching the same numbers for every chunk size."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle.softmax import softmax_rows


def test_matches_scipy():
    x = np.random.default_rng(0).standard_normal((7, 33)) * 5
    y, lse = softmax_rows(x)
    np.testing.assert_allclose(y, softmax(x, axis=-1), rtol=1e-13, atol=0)
    np.testing.assert_allclose(lse, logsumexp(x, axis=-1), rtol=1e-14, atol=0)


def test_rows_sum_to_one_and_shift_invariance():
    x = np.random.default_rng(1).standard_normal((5, 100)) * 30
    y, lse = softmax_rows(x)
    np.testing.assert_allclose(y.sum(-1), 1.0, atol=1e-14)
    y2, lse2 = softmax_rows(x + 123.25)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(lse2, lse + 123.25, rtol=1e-14)


def test_closed_forms():
    y, lse = softmax_rows(np.full((1, 8), 3.0))
    np.testing.assert_allclose(y, 1 / 8, rtol=1e-15)
    np.testing.assert_allclose(lse, 3.0 + np.log(8.0), rtol=1e-15)
    a, b = 0.75, -1.5
    y, _ = softmax_rows(np.array([[a, b]]))
    np.testing.assert_allclose(y[0, 0], 1.0 / (1.0 + np.exp(b - a)), rtol=1e-15)


def test_empty_and_partly_masked_rows():
    x = np.array([[-np.inf, -np.inf, -np.inf], [-np.inf, 2.0, -np.inf]])
    y, lse = softmax_rows(x)
    assert np.all(y[0] == 0) and np.isneginf(lse[0])
    np.testing.assert_array_equal(y[1], [0.0, 1.0, 0.0])
    assert lse[1] == 2.0


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 64])
def test_two_read_recurrence_reaches_the_definition(chunk):
    # read 1 of the guide: d_k = max(d_{k-1}, max chunk k), s_k = s_{k-1} e^(d_{k-1}-d_k) + sum e^(a-d_k)
    x = np.random.default_rng(2).standard_normal(50) * 8
    d, s = -np.inf, 0.0
    for c0 in range(0, x.size, chunk):
        c = x[c0:c0 + chunk]
        dn = max(d, c.max())
        s = s * np.exp(d - dn) + np.exp(c - dn).sum()
        d = dn
    y_two = np.exp(x - d) / s                      # read 2
    y, lse = softmax_rows(x[None, :])
    np.testing.assert_allclose(y_two, y[0], rtol=1e-13)
    np.testing.assert_allclose(d + np.log(s), lse[0], rtol=1e-14)
