"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only the tests, the package smoke check and the CPU-baseline leg of the
benchmark use it. It shares no code with the CUDA library.

What it computes, and where that is defined
--------------------------------------------
"NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention ..."
(quidproquo.cc), section "Intuition: the naive way makes many warehouse trips":
for one query q, the scores are a_i = q . k_i; the maximum Amax is found, each
score is exponentiated as exp(a_i - Amax), the exponentials are summed into a
denominator S, divided by S to give the weights, and the output is the
weighted sum of the rows of v.  The same page, "Mechanism" and "Expand: the
correction for the output O", states that the one-pass FlashAttention
recurrence reaches exactly this result; "6.3 FlashAttention" (comfyai.app),
section "6.3.2 Standard Attention and Safe Softmax", gives the same
max-subtracted ("safe") softmax.  So the oracle is this definition, in the
order the guide lists, one step per line:

    a      = scale * (q_rows @ k^T)          materialise the scores
    a[m]   = -inf   where masked              causal: key j visible iff j <= i
    Amax   = max_j a                          row maximum
    e      = exp(a - Amax)                    safe exponentials
    S      = sum_j e                          denominator
    w      = e / S                            attention weights
    O      = w @ v                            weighted sum of the values
    LSE    = Amax + ln S                      natural-log log-sum-exp

The pages scale the scores only implicitly (the softmax of q . k); the scale
factor and the causal mask rule ("key j visible to query i iff j <= i") are
the workload's, and the log-sum-exp is the natural-log summary m + ln l of the
two per-row statistics m (max) and l (sum) that "6.3 FlashAttention" keeps for
each query row.  A matrix product (numpy/BLAS, fp64) is used as a library step
for q @ k^T and w @ v; nothing is blocked, fused or reordered beyond that.

Inputs are taken exactly: bf16 tensors are widened to fp64 (an exact
conversion), so the oracle sees the very values the GPU sees.
"""
from __future__ import annotations

import numpy as np

__all__ = ["to_f64", "attention_rows", "attention_head", "attention"]


def to_f64(x) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype, incl. bf16) or an
    array-like to a float64 numpy array."""
    if hasattr(x, "detach"):  # torch tensor, imported lazily by the caller
        import torch

        return x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def attention_rows(q_rows, k, v, scale, causal=False, row_index=None,
                   return_weights=False):
    """Attention for a set of query rows of ONE head, in fp64.

    q_rows    : [R, D] query rows
    k, v      : [Lk, D] keys and values of that head
    scale     : score scale (a = scale * q . k)
    causal    : if true, row r may see key j only when j <= row_index[r]
    row_index : [R] position i of each query row (needed when causal)

    Returns (O [R, D], LSE [R]) and, if asked, the weights w [R, Lk].
    A row whose keys are all masked returns O = 0 and LSE = -inf (this cannot
    happen for the causal rule j <= i, since key 0 is always visible).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, Lk = q_rows.shape[0], k.shape[0]

    # 1. materialise the scores a_ij = scale * q_i . k_j
    a = float(scale) * (q_rows @ k.T)

    # 2. causal mask: key j is visible to query i iff j <= i
    if causal:
        if row_index is None:
            raise ValueError("causal attention needs row_index")
        i = np.asarray(row_index, dtype=np.int64).reshape(R, 1)
        j = np.arange(Lk, dtype=np.int64).reshape(1, Lk)
        a = np.where(j <= i, a, -np.inf)

    # 3. row maximum Amax
    amax = a.max(axis=1)
    empty = ~np.isfinite(amax)
    amax_safe = np.where(empty, 0.0, amax)

    # 4. safe exponentials exp(a - Amax)
    e = np.exp(a - amax_safe[:, None])

    # 5. denominator S
    s = e.sum(axis=1)

    # 6. weights w = e / S
    s_safe = np.where(empty, 1.0, s)
    w = e / s_safe[:, None]

    # 7. weighted sum of the values
    o = w @ v

    # 8. log-sum-exp in natural log
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, amax_safe + np.log(s_safe))

    if return_weights:
        return o, lse, w
    return o, lse


def attention_head(q, k, v, scale, causal=False, rows=None, chunk=256):
    """All (or the selected) query rows of one head, processed in chunks of
    rows so that the materialised score block stays bounded in memory.

    q: [Lq, D], k, v: [Lk, D]; rows: optional 1-D array of query positions.
    Returns (O [R, D], LSE [R]) in the order of `rows` (or 0..Lq-1).
    """
    q = np.asarray(q, dtype=np.float64)
    if rows is None:
        rows = np.arange(q.shape[0], dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    o = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.empty(rows.shape[0], dtype=np.float64)
    for c0 in range(0, rows.shape[0], chunk):
        r = rows[c0:c0 + chunk]
        o[c0:c0 + chunk], lse[c0:c0 + chunk] = attention_rows(
            q[r], k, v, scale, causal=causal, row_index=r)
    return o, lse


def attention(q, k, v, scale, causal=False):
    """Full attention over [B, H, L, D] inputs. Returns O [B,H,Lq,D] and
    LSE [B,H,Lq] in fp64. Meant for small shapes."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, H, Lq, D = q.shape
    o = np.empty((B, H, Lq, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, Lq), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h],
                                                scale, causal=causal)
    return o, lse
