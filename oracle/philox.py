"""Philox counter-based random numbers, written from their published definition.

TEST INFRASTRUCTURE ONLY (like the rest of this folder): only the tests, the
package smoke check and the benchmark's CPU legs may import it; it shares no
code with the CUDA library.

Definition followed: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011), section 3.2
("Philox"): a keyed bijection of a counter of four W-bit words, built from R
rounds.  Each round multiplies two of the words by fixed odd constants
(M0, M1), keeps both halves of the double-width products, and permutes and
xors them with the other two words and the round key:

    (hi0, lo0) = M0 * x0          (hi1, lo1) = M1 * x2
    x0' = hi1 ^ x1 ^ k0           x1' = lo1
    x2' = hi0 ^ x3 ^ k1           x3' = lo0

and the key is bumped by the Weyl constants (W0, W1) between rounds.  The
paper's recommended instances are Philox-4x32-10 and Philox-4x64-10; the
constants below are the published ones for each width.  One generic routine
serves both widths, so the 64-bit instance (checked in the tests against
numpy's library implementation, numpy.random.Philox) pins the round
structure, the word order and the key schedule that the 32-bit instance
shares.

The dropout contract of the attention library draws its bits from
Philox-4x32-10; see oracle/dropout.py.
"""
from __future__ import annotations

import numpy as np

__all__ = ["PHILOX_CONSTANTS", "philox", "philox4x32_10", "philox4x64_10"]

# width -> (M0, M1, W0, W1)
PHILOX_CONSTANTS = {
    32: (0xD2511F53, 0xCD9E8D57, 0x9E3779B9, 0xBB67AE85),
    64: (0xD2E7470EE14C6C93, 0xCA5A826395121157, 0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B),
}


def philox(ctr, key, width: int, rounds: int = 10):
    """Philox-4xW-R on Python integers: ctr = 4 words, key = 2 words, each
    below 2**width.  Returns the 4 output words."""
    m0, m1, w0, w1 = PHILOX_CONSTANTS[width]
    mask = (1 << width) - 1
    x = [int(c) & mask for c in ctr]
    k0, k1 = (int(k) & mask for k in key)
    for _ in range(rounds):
        p0 = m0 * x[0]
        p1 = m1 * x[2]
        x = [((p1 >> width) ^ x[1] ^ k0) & mask, p1 & mask,
             ((p0 >> width) ^ x[3] ^ k1) & mask, p0 & mask]
        k0 = (k0 + w0) & mask
        k1 = (k1 + w1) & mask
    return x


def philox4x64_10(ctr, key):
    return philox(ctr, key, 64, 10)


def philox4x32_10(ctr, key):
    """Philox-4x32-10.  Scalar words, or numpy integer arrays of one shape
    (all four counter words broadcast together) for many counters at once;
    returns four uint32 arrays in the array case."""
    if all(np.isscalar(c) for c in ctr) and all(np.isscalar(k) for k in key):
        return philox(ctr, key, 32, 10)
    m0, m1, w0, w1 = (np.uint64(c) for c in PHILOX_CONSTANTS[32])
    lo32 = np.uint64(0xFFFFFFFF)
    sh = np.uint64(32)
    x = [np.asarray(c, dtype=np.uint64) & lo32 for c in ctr]
    x = np.broadcast_arrays(*x)
    x = [a.copy() for a in x]
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = m0 * x[0]          # < 2**64: exact in uint64
        p1 = m1 * x[2]
        x = [((p1 >> sh) ^ x[1] ^ k0) & lo32, p1 & lo32, ((p0 >> sh) ^ x[3] ^ k1) & lo32, p0 & lo32]
        k0 = (k0 + w0) & lo32
        k1 = (k1 + w1) & lo32
    return [a.astype(np.uint32) for a in x]
