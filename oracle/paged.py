"""fp64 CPU oracle for single-query attention against a paged key/value cache.

TEST INFRASTRUCTURE ONLY (like oracle.naive): only the tests, the package
smoke check and the benchmark's CPU legs may import it; it shares no code with
the CUDA library.

What it computes
----------------
"NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention"
(quidproquo.cc) splits generation into prefill and decode ("For any speed-up,
ask what it costs", slide 5) and leaves the cache that decode reads to the
next part of the lecture ("Back to real models: you are probably using it
already", last paragraphs).  The pages fix no cache layout, so this is the
plainest paged reading, the same one include/fa.h documents: the cached keys
and values of sequence b are its positions 0 .. seq_lens[b]-1, in order;
position p sits in page block_table[b, p // page_size], row p % page_size, of
caches shaped [num_pages, page_size, H, D].  Decode attention for sequence b
and head h is then the plain definition of oracle.naive (one query row, all
of that sequence's positions visible) on the gathered keys and values.

A length is clamped to [0, max_pages_per_seq * page_size]; a sequence of
length 0 has no visible key and gets O = 0, LSE = -inf (the empty-row
convention of oracle.naive).
"""
from __future__ import annotations

import numpy as np

from .naive import attention_rows, to_f64

__all__ = ["gather_sequence", "decode_paged"]


def gather_sequence(k_cache, v_cache, table_row, length, page_size):
    """Keys and values [L, H, D] of one sequence, position by position."""
    p = np.arange(length, dtype=np.int64)
    pages = np.asarray(table_row, dtype=np.int64)[p // page_size]
    rows = p % page_size
    return k_cache[pages, rows], v_cache[pages, rows]


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale):
    """q [B, H, D] (or [B, H, 1, D]); caches [num_pages, page_size, H, D];
    block_table [B, max_pages]; seq_lens [B].  Returns O [B, H, D] and
    LSE [B, H] in fp64."""
    q = to_f64(q)
    if q.ndim == 4:
        q = q[:, :, 0, :]
    kc, vc = to_f64(k_cache), to_f64(v_cache)
    bt = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table, dtype=np.int64)
    lens = np.asarray(seq_lens.cpu() if hasattr(seq_lens, "cpu") else seq_lens, dtype=np.int64)
    B, H, D = q.shape
    page_size = kc.shape[1]
    cap = bt.shape[1] * page_size
    o = np.zeros((B, H, vc.shape[-1]), dtype=np.float64)
    lse = np.full((B, H), -np.inf, dtype=np.float64)
    for b in range(B):
        length = int(min(max(lens[b], 0), cap))
        if length == 0:
            continue
        kb, vb = gather_sequence(kc, vc, bt[b], length, page_size)
        for h in range(H):
            ob, lb = attention_rows(q[b, h][None, :], kb[:, h, :], vb[:, h, :], scale)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse
