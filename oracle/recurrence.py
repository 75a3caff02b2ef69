"""The guide's chunk-by-chunk online-softmax recurrence, in fp64.

TEST INFRASTRUCTURE ONLY (like the rest of this folder). It is not the
oracle: it exists so that the tests can pin the oracle (a two-pass
definition) against the one-pass derivation on the pages.

Source: "NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash
Attention ..." (quidproquo.cc), sections "Expand: why multiplying by
exp(d1 - d2) fixes it" and "Expand: the correction for the output O".  For
one query, keys split into chunks 1..B, with d the running maximum, s the
running denominator and O the running output, the guide's update for chunk k
is

    d_k = max(d_{k-1}, max of chunk k)
    s_k = s_{k-1} * exp(d_{k-1} - d_k) + sum_{i in chunk k} exp(a_i - d_k)
    O_k = O_{k-1} * (s_{k-1} / s_k) * exp(d_{k-1} - d_k)
          + sum_{i in chunk k} [exp(a_i - d_k) / s_k] * v_i

and after the last chunk d_B = Amax, s_B is the full denominator and
O_B = sum_i softmax(a)_i v_i.  The first chunk starts from d_0 = -inf,
s_0 = 0, O_0 = 0 (the guide starts by taking chunk 1's maximum as d_1); the
terms multiplied by s_0 = 0 are dropped for k = 1 so that exp(-inf + inf) is
never formed.

"6.3 FlashAttention" (comfyai.app), "A Simple Example", walks the same merge
on the vector [1, 2, 3, 4] split into [1, 2] and [3, 4].
"""
from __future__ import annotations

import numpy as np

__all__ = ["rescale_identity_sides", "online_softmax_stats", "online_attention_row"]


def rescale_identity_sides(a_chunk, d1, d2):
    """Both sides of the guide's rescale identity for one chunk:
    s1 * exp(d1 - d2) and sum_i exp(a_i - d2), where s1 = sum_i exp(a_i - d1).
    """
    a = np.asarray(a_chunk, dtype=np.float64)
    s1 = np.exp(a - d1).sum()
    return s1 * np.exp(d1 - d2), np.exp(a - d2).sum()


def online_softmax_stats(a, chunk):
    """Runs the (d_k, s_k) recurrence over `a` in chunks of `chunk` entries.
    Returns the list of (d_k, s_k) after every chunk."""
    a = np.asarray(a, dtype=np.float64)
    out = []
    d_prev, s_prev = -np.inf, 0.0
    for c0 in range(0, a.shape[0], chunk):
        blk = a[c0:c0 + chunk]
        d_k = max(d_prev, blk.max())
        local = np.exp(blk - d_k).sum()
        if c0 == 0:
            s_k = local
        else:
            s_k = s_prev * np.exp(d_prev - d_k) + local
        out.append((d_k, s_k))
        d_prev, s_prev = d_k, s_k
    return out


def online_attention_row(q, k, v, scale, chunk, n_visible=None):
    """One query row by the guide's one-pass recurrence for d, s and O.

    q: [D], k, v: [L, D]. Only the first n_visible keys are used (all when
    None), which is how a causal row i sees keys 0..i.
    Returns (O [D], d_B, s_B) so that LSE = d_B + ln s_B.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L = k.shape[0] if n_visible is None else int(n_visible)
    d_prev, s_prev = -np.inf, 0.0
    o_prev = np.zeros(v.shape[1], dtype=np.float64)
    for c0 in range(0, L, chunk):
        c1 = min(c0 + chunk, L)
        a = float(scale) * (k[c0:c1] @ q)          # a_i = q . k_i for the chunk
        d_k = max(d_prev, a.max())
        e = np.exp(a - d_k)
        if c0 == 0:
            s_k = e.sum()
            o_k = (e / s_k) @ v[c0:c1]
        else:
            s_k = s_prev * np.exp(d_prev - d_k) + e.sum()
            o_k = (o_prev * (s_prev / s_k) * np.exp(d_prev - d_k)
                   + (e / s_k) @ v[c0:c1])
        d_prev, s_prev, o_prev = d_k, s_k, o_k
    return o_prev, d_prev, s_prev
