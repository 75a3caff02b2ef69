"""fp64 CPU oracle for attention with dropout on the weights (fa_fwd_dropout).

TEST INFRASTRUCTURE ONLY (like oracle.naive): only the tests, the package
smoke check and the benchmark's CPU legs may import it; it shares no code with
the CUDA library.

What it computes
----------------
"6.3 FlashAttention" (comfyai.app), section "6.3.3 FlashAttention Forward
Process", parts "Difficulty of Tiling" and "Kernel Fusion": training-time
attention is matrix multiplication -> scale -> mask -> softmax -> dropout ->
matrix multiplication, and the mask and the dropout are fused into the work on
each tile, in on-chip memory.  The pages give no formula for the dropout step
and no random number contract, so this library fixes its own (a reading,
stated here and in the design notes):

  * dropout acts on the normalised softmax weights w (after masking): each
    weight is kept with probability 1 - p and scaled by 1 / (1 - p), or set to
    0, so E[output] = softmax(..) v; the log-sum-exp is that of the undropped
    scores (dropout does not change the softmax statistics);
  * the drop probability is quantised to t / 256 with t = floor(256 p + 0.5)
    (0 <= t <= 255), computed in double precision; the kept weights are
    scaled by 256 / (256 - t), which keeps the output unbiased;
  * the bits come from Philox-4x32-10 (oracle.philox) with key
    (seed mod 2^32, seed div 2^32) and counter (j div 16, i, b*H + h, offset)
    for key position j of query row i in head h of batch b; the call returns
    four 32-bit words x0..x3, and key j takes byte (j mod 4) of word
    x_((j div 4) mod 4), little-endian (bits 8 (j mod 4) .. 8 (j mod 4) + 7);
  * key j is kept iff that byte >= t.

So, for one head, in the order of the pages' steps:

    a    = scale * q k^T                 scores
    a[m] = -inf where masked             causal: key j visible iff j <= i
    w    = softmax(a) row by row         (oracle.naive's definition)
    z    = keep mask from the contract above
    O    = ((w * z) @ v) * 256 / (256 - t)
    LSE  = log-sum-exp of a              (unchanged by dropout)

The backward (fa_bwd_dropout) is the gradient of <dO, O> for that forward,
with the keep mask z fixed (it depends on the seed, not on q, k, v); with
s = 256 / (256 - t), step by step:

    dV  = s (w * z)^T dO
    dWz = dO v^T                         gradient of the dropped weights
    dW  = s z * dWz                      gradient of the weights w
    dA  = w * (dW - rowsum(w * dW))      softmax's Jacobian
    dQ  = scale dA k,   dK = scale dA^T q

(rowsum(w * dW) equals rowsum(dO * O) with O the dropout forward's output,
the quantity FlashAttention-style backward passes compute once per row.)
"""
from __future__ import annotations

import math

import numpy as np

from oracle.naive import attention_rows
from oracle.philox import philox4x32_10

__all__ = ["drop_threshold", "keep_mask", "attention_dropout_rows", "attention_dropout",
           "backward_dropout_head", "backward_dropout"]


def drop_threshold(p_drop: float) -> int:
    """t = floor(256 p + 0.5) in double precision; the byte threshold."""
    p = float(np.float32(p_drop))  # the C ABI takes p as a 32-bit float
    if not (0.0 <= p < 1.0) or not math.isfinite(p):
        raise ValueError("p_drop must be in [0, 1)")
    t = int(math.floor(p * 256.0 + 0.5))
    if t > 255:
        raise ValueError("p_drop rounds to 256/256")
    return t


def keep_mask(bh: int, rows, Lk: int, t: int, seed: int, offset: int) -> np.ndarray:
    """Boolean [len(rows), Lk]: key j of query row rows[r] in head bh kept."""
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    groups = np.arange((Lk + 15) // 16, dtype=np.uint64).reshape(1, -1)
    seed = int(seed) & ((1 << 64) - 1)
    key = (seed & 0xFFFFFFFF, seed >> 32)
    x = philox4x32_10((groups, rows, np.uint64(bh), np.uint64(int(offset) & 0xFFFFFFFF)), key)
    words = np.stack(x, axis=-1)                      # [R, G, 4] uint32
    b = words.view(np.uint8).reshape(words.shape[0], -1)  # little-endian bytes: [R, 16 G]
    b = b[:, :Lk]
    return b >= np.uint8(t) if t > 0 else np.ones(b.shape, dtype=bool)


def attention_dropout_rows(q_rows, k, v, scale, causal, row_index, bh, p_drop, seed, offset):
    """Attention with dropout for query rows `row_index` of head `bh`.
    Returns (O [R, D], LSE [R], keep [R, Lk])."""
    t = drop_threshold(p_drop)
    row_index = np.asarray(row_index)
    # scores, scale, mask and softmax: the plain oracle's definition
    _, lse, w = attention_rows(q_rows, k, v, scale, causal=causal, row_index=row_index,
                               return_weights=True)
    z = keep_mask(bh, row_index, np.asarray(k).shape[0], t, seed, offset)
    o = ((w * z) @ np.asarray(v, dtype=np.float64)) * (256.0 / (256.0 - t))
    return o, lse, z


def attention_dropout(q, k, v, scale, causal, p_drop, seed, offset):
    """Whole tensors [B, H, L, D] (numpy fp64 or exact widenings of bf16)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Lq, D = q.shape
    O = np.zeros((B, H, Lq, v.shape[-1]))
    LSE = np.zeros((B, H, Lq))
    rows = np.arange(Lq)
    for b in range(B):
        for h in range(H):
            O[b, h], LSE[b, h], _ = attention_dropout_rows(q[b, h], k[b, h], v[b, h], scale, causal, rows,
                                                           b * H + h, p_drop, seed, offset)
    return O, LSE


def backward_dropout_head(q, k, v, do, scale, causal, bh, p_drop, seed, offset):
    """Gradients of <dO, O> for one head of the dropout forward (head index bh
    in the counter): q, do [Lq, D]; k, v [Lk, D].  Returns dq, dk, dv (fp64)."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    t = drop_threshold(p_drop)
    s = 256.0 / (256.0 - t)
    rows = np.arange(q.shape[0])
    _, _, w = attention_rows(q, k, v, scale, causal=causal, row_index=rows, return_weights=True)
    z = keep_mask(bh, rows, k.shape[0], t, seed, offset).astype(np.float64)
    dv = s * ((w * z).T @ do)
    dwz = do @ v.T
    dw = s * z * dwz
    da = w * (dw - (w * dw).sum(axis=1, keepdims=True))
    dq = float(scale) * (da @ k)
    dk = float(scale) * (da.T @ q)
    return dq, dk, dv


def backward_dropout(q, k, v, do, scale, causal, p_drop, seed, offset):
    """[B, H, L, D] inputs (exact widenings of bf16 or fp64).  Returns dq, dk,
    dv as fp64 arrays of the inputs' shapes.  Meant for small shapes."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_dropout_head(q[b, h], k[b, h], v[b, h], do[b, h], scale,
                                                                 causal, b * H + h, p_drop, seed, offset)
    return dq, dk, dv
