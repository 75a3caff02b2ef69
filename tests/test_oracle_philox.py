"""Pins the oracle's 32-bit Philox (oracle.philox.philox4x32_10) to an
independent library implementation of the same generator.

The dropout contract draws its bits from Philox-4x32-10 (Salmon, Moraes, Dror
and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011, section
3.2).  The oracle's 64-bit instance is checked against numpy's Philox-4x64-10
elsewhere; nothing there fixes the 32-bit instance's own constants (two
multipliers, two Weyl increments).  Here the 32-bit instance is compared word
for word with Triton's ``philox_impl`` (a library routine by other authors,
run on the CPU through Triton's interpreter in a child process) on counters
and keys that exercise every word: zeros, all-ones, the hexadecimal digits of
pi, random words, and counters shaped like the dropout contract's
(j div 16, i, b*H + h, offset) with keys split from 64-bit seeds.  A planted
mistake in each constant, and in the output word order, must make the
comparison fail.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import philox as ph

HERE = os.path.dirname(os.path.abspath(__file__))
PI_WORDS = (0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344, 0xA4093822, 0x299F31D0)


def _cases():
    ctr, key = [], []
    ctr.append((0, 0, 0, 0)); key.append((0, 0))
    m = 0xFFFFFFFF
    ctr.append((m, m, m, m)); key.append((m, m))
    ctr.append(PI_WORDS[:4]); key.append(PI_WORDS[4:])
    rng = np.random.default_rng(20111112)
    for _ in range(96):
        w = [int(x) for x in rng.integers(0, 1 << 32, size=6, dtype=np.uint64)]
        ctr.append(tuple(w[:4])); key.append(tuple(w[4:]))
    # the dropout contract's counters: (key block j div 16, query row, head, offset)
    for seed in (1234, (1 << 40) + 17, 0x123456789ABCDEF0):
        for (jb, i, bh, off) in ((0, 0, 0, 0), (8, 127, 5, 0), (511, 8191, 63, 0),
                                 (17, 4095, 31, 123456), (4095, 65535, 0, 3)):
            ctr.append((jb, i, bh, off)); key.append((seed & m, seed >> 32))
    return ctr, key


@pytest.fixture(scope="module")
def triton_words():
    pytest.importorskip("triton")
    ctr, key = _cases()
    req = json.dumps({"ctr": [list(c) for c in ctr], "key": [list(k) for k in key]})
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "philox_triton_ref.py")], input=req,
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.fail(f"Triton's Philox did not run on the CPU interpreter:\n{r.stderr[-2000:]}")
    reply = json.loads(r.stdout)
    return ctr, key, reply["words"]


def test_scalar_instance_matches_triton(triton_words):
    ctr, key, words = triton_words
    for c, k, w in zip(ctr, key, words):
        assert ph.philox4x32_10(c, k) == w, (c, k)


def test_array_instance_matches_triton(triton_words):
    ctr, key, words = triton_words
    # the numpy path takes one key per call: group the counters by key
    by_key = {}
    for idx, k in enumerate(key):
        by_key.setdefault(tuple(k), []).append(idx)
    for k, idxs in by_key.items():
        cols = [np.array([ctr[i][c] for i in idxs], dtype=np.uint64) for c in range(4)]
        got = ph.philox4x32_10(cols, k)
        for r, i in enumerate(idxs):
            assert [int(g[r]) for g in got] == words[i], (ctr[i], k)


def test_zero_counter_zero_key_words(triton_words):
    # the all-zero input is where a word-order or round-structure slip shows
    # first; both implementations must give four distinct nonzero words
    _, _, words = triton_words
    assert len(set(words[0])) == 4 and all(w != 0 for w in words[0])


@pytest.mark.parametrize("which", range(4))
def test_a_wrong_constant_is_caught(triton_words, which, monkeypatch):
    ctr, key, words = triton_words
    consts = list(ph.PHILOX_CONSTANTS[32])
    consts[which] ^= 1 << 7            # one flipped bit in M0, M1, W0 or W1
    monkeypatch.setitem(ph.PHILOX_CONSTANTS, 32, tuple(consts))
    mismatches = sum(ph.philox(c, k, 32, 10) != w for c, k, w in zip(ctr, key, words))
    assert mismatches > 0.9 * len(ctr)


def test_swapped_multipliers_and_word_order_are_caught(triton_words, monkeypatch):
    ctr, key, words = triton_words
    m0, m1, w0, w1 = ph.PHILOX_CONSTANTS[32]
    monkeypatch.setitem(ph.PHILOX_CONSTANTS, 32, (m1, m0, w0, w1))
    assert all(ph.philox(c, k, 32, 10) != w for c, k, w in zip(ctr, key, words))
    monkeypatch.setitem(ph.PHILOX_CONSTANTS, 32, (m0, m1, w0, w1))
    # outputs in reversed order, or nine rounds instead of ten
    assert all(ph.philox(c, k, 32, 10)[::-1] != w for c, k, w in zip(ctr, key, words))
    assert all(ph.philox(c, k, 32, 9) != w for c, k, w in zip(ctr, key, words))
