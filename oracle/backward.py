"""fp64 CPU oracle for the attention backward pass (dQ, dK, dV).

TEST INFRASTRUCTURE ONLY (like oracle.naive); it shares no code with the CUDA
library.

"6.3 FlashAttention" (comfyai.app), "A simple implementation w/ C++" (last
paragraph) and "Computation and GPU Memory": for training, the intermediate
results of the forward pass are not saved but recomputed during the backward
pass, at the cost of extra FLOPs.  The pages give no backward formulas, so
the oracle is the plain definition of what a backward pass returns: the
gradients of the scalar <dO, O> with respect to q, k and v, where
O = softmax(scale q k^T [causal mask]) v is the forward of oracle.naive, for
every head.  Written out step by step in fp64:

    A   = scale * q k^T  (masked entries -inf)      scores
    P   = exp(A - rowmax) / rowsum                   weights (safe softmax)
    dV  = P^T dO                                     O = P V
    dP  = dO V^T
    dA  = P * (dP - rowsum(P * dP))                  softmax's Jacobian
    dQ  = scale * dA k,   dK = scale * dA^T q        A = scale q k^T

(rowsum(P * dP) equals rowsum(dO * O), the quantity FlashAttention's
backward uses; the oracle takes the first form.)  A matrix product is a
library step.
"""
from __future__ import annotations

import numpy as np

from .naive import to_f64

__all__ = ["backward_head", "backward"]


def backward_head(q, k, v, do, scale, causal=False):
    """One head: q, do [Lq, D]; k, v [Lk, D].  Returns dq, dk, dv (fp64)."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    Lq, Lk = q.shape[0], k.shape[0]
    a = float(scale) * (q @ k.T)
    if causal:
        i = np.arange(Lq).reshape(Lq, 1)
        j = np.arange(Lk).reshape(1, Lk)
        a = np.where(j <= i, a, -np.inf)
    amax = a.max(axis=1, keepdims=True)
    e = np.exp(a - amax)
    p = e / e.sum(axis=1, keepdims=True)
    dv = p.T @ do
    dp = do @ v.T
    da = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    dq = float(scale) * (da @ k)
    dk = float(scale) * (da.T @ q)
    return dq, dk, dv


def backward(q, k, v, do, scale, causal=False):
    """[B, H, L, D] inputs (any float type, widened exactly).  Returns dq, dk,
    dv as fp64 arrays of the inputs' shapes.  Meant for small shapes."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h],
                                                         scale, causal)
    return dq, dk, dv
