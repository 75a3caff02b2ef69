"""fp64 CPU oracle for the row softmax (fa_softmax_rows).

TEST INFRASTRUCTURE ONLY (like oracle.naive); it shares no code with the CUDA
library.

"NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention"
(quidproquo.cc), "Intuition: the naive way makes many warehouse trips": the
weights of a row a_1..a_N are found by taking the maximum Amax, the
exponentials exp(a_i - Amax), their sum S, and dividing: a_hat_i =
exp(a_i - Amax) / S.  The two-read order of "Expand: why multiplying by
exp(d1 - d2) fixes it" reaches the same numbers; the oracle is the plain
definition, step by step, in fp64.  A row of only -inf has no weights: the
oracle returns 0 and a log-sum-exp of -inf (the empty-row convention of
oracle.naive).
"""
from __future__ import annotations

import numpy as np

__all__ = ["softmax_rows"]


def softmax_rows(x):
    """x: [..., N] (any float type, widened exactly to fp64).
    Returns (y, lse): y[..., i] = exp(x_i - Amax) / S, lse = Amax + ln S."""
    x = np.asarray(x, dtype=np.float64)
    amax = x.max(axis=-1, keepdims=True)                      # Amax
    empty = ~np.isfinite(amax)
    amax_safe = np.where(empty, 0.0, amax)
    e = np.exp(x - amax_safe)                                 # exp(a_i - Amax)
    s = e.sum(axis=-1, keepdims=True)                         # S
    s_safe = np.where(empty, 1.0, s)
    y = np.where(empty, 0.0, e / s_safe)                      # a_hat_i
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, amax_safe + np.log(s_safe))[..., 0]
    return y, lse
