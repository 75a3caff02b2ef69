"""The library's device Philox-4x32-10 (csrc/philox.cuh, the routine the
dropout kernels call) against the CPU oracle, bit for bit.

The oracle's 32-bit Philox is pinned to Triton's independent implementation
(tests/test_oracle_philox.py); here a test-only probe kernel
(tests/philox_probe.cu) runs the library's own routines (one counter; two
counters under one key with their rounds interleaved; and the row forms that
fold the parts of the first two rounds shared by one query row's calls and
take the later rounds' keys precomputed, and the column form that folds
the parts shared by one key block's calls across query rows) on the same counters and keys, plus
random ones and counters shaped like the dropout contract's, and every output
word must agree.  The same probe runs the kernels' keep masks (four random
bytes against the threshold t at once, as 16-bit pair masks and as 32-bit
per-key masks) for every t and every byte value, against the plain
comparison byte >= t.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from exact_attention_03_gb300 import build as fa_build
from oracle.philox import philox4x32_10
from test_oracle_philox import _cases

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    os.makedirs(fa_build.BUILD_DIR, exist_ok=True)
    so = os.path.join(fa_build.BUILD_DIR, "libphilox_probe.so")
    cmd = [fa_build.nvcc(), *fa_build.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", fa_build.CSRC, os.path.join(HERE, "philox_probe.cu"), "-o", so]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(so)
    lib.philox_probe.restype = ctypes.c_int
    lib.philox_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    return lib


def _run(lib, recs, mode=0):
    recs = np.ascontiguousarray(recs, dtype=np.uint32)
    out = np.zeros((recs.shape[0], 4), dtype=np.uint32)
    assert lib.philox_probe(recs.ctypes.data, out.ctypes.data, recs.shape[0], mode) == 0
    return out


def _oracle(recs):
    out = np.zeros((recs.shape[0], 4), dtype=np.uint32)
    keys = {}
    for i, r in enumerate(recs):
        keys.setdefault((int(r[4]), int(r[5])), []).append(i)
    for k, idx in keys.items():
        idx = np.array(idx)
        w = philox4x32_10([recs[idx, c].astype(np.uint64) for c in range(4)], k)
        out[idx] = np.stack(w, axis=1)
    return out


def test_device_philox_matches_oracle_on_the_pinned_cases(probe):
    ctr, key = _cases()
    recs = np.array([list(c) + list(k) for c, k in zip(ctr, key)], dtype=np.uint64)
    got = _run(probe, recs)
    want = np.array([philox4x32_10(c, k) for c, k in zip(ctr, key)], dtype=np.uint32)
    assert np.array_equal(got, want)


def test_device_philox_matches_oracle_on_random_and_contract_counters(probe):
    rng = np.random.default_rng(5)
    n = 1 << 16
    recs = rng.integers(0, 1 << 32, size=(n, 6), dtype=np.uint64)
    recs[:, 4:] = recs[:8, 4:][np.arange(n) % 8]          # eight keys
    # the contract's counters: (j div 16 for keys up to 65536, row, head, offset)
    m = n // 2
    recs[:m, 0] = rng.integers(0, 4096, size=m)
    recs[:m, 1] = rng.integers(0, 65536, size=m)
    recs[:m, 2] = rng.integers(0, 512, size=m)
    recs[:m, 3] = rng.choice([0, 1, 123456], size=m)
    assert np.array_equal(_run(probe, recs), _oracle(recs))


def test_paired_device_philox_matches_oracle(probe):
    # the two-counter routine the D = 128 dropout kernels use: records 2m and
    # 2m+1 share a key, as the two 16-key groups of a 32-key block do
    rng = np.random.default_rng(6)
    n = 1 << 14
    recs = rng.integers(0, 1 << 32, size=(n, 6), dtype=np.uint64)
    recs[1::2, 4:] = recs[0::2, 4:]
    recs[0::2, 0] = rng.integers(0, 4096, size=n // 2)
    recs[1::2, 0] = recs[0::2, 0] + 1
    recs[1::2, 1:4] = recs[0::2, 1:4]
    assert np.array_equal(_run(probe, recs, mode=1), _oracle(recs))


@pytest.mark.parametrize("paired", [False, True])
def test_row_device_philox_matches_oracle(probe, paired):
    # the row routines the dropout kernels use: words 1-3 (query row, head,
    # offset) and the key are fixed per row, the key block j div 16 varies
    rng = np.random.default_rng(7 + paired)
    n = 1 << 14
    recs = rng.integers(0, 1 << 32, size=(n, 6), dtype=np.uint64)
    recs[:n // 2, 0] = rng.integers(0, 4096, size=n // 2)
    if paired:
        recs[1::2, 1:] = recs[0::2, 1:]
    assert np.array_equal(_run(probe, recs, mode=3 if paired else 2), _oracle(recs))


def test_column_device_philox_matches_oracle(probe):
    # the column routine of the dropout backward's key-block kernel: word 0
    # (the key block j div 16), head, offset and key fixed per column, the
    # query row (word 1) varying
    rng = np.random.default_rng(9)
    n = 1 << 14
    recs = rng.integers(0, 1 << 32, size=(n, 6), dtype=np.uint64)
    recs[:n // 2, 0] = rng.integers(0, 4096, size=n // 2)
    recs[:n // 2, 1] = rng.integers(0, 65536, size=n // 2)
    recs[:n // 2, 2] = rng.integers(0, 512, size=n // 2)
    assert np.array_equal(_run(probe, recs, mode=5), _oracle(recs))


def test_keep_masks_match_the_byte_comparison_for_every_threshold(probe):
    # every byte value in every position, for every threshold t = 0..255
    vals = np.arange(256, dtype=np.uint64)
    words = np.concatenate([vals * 0x01010101,                       # all four bytes equal
                            vals | ((255 - vals) << 8) | (((vals * 7) % 256) << 16) | (((vals * 13 + 5) % 256) << 24)])
    recs = np.zeros((256 * len(words), 6), dtype=np.uint64)
    recs[:, 0] = np.tile(words, 256)
    recs[:, 1] = np.repeat(np.arange(256, dtype=np.uint64), len(words))
    got = _run(probe, recs, mode=4)
    w = recs[:, 0].astype(np.uint32)
    t = recs[:, 1].astype(np.uint32)
    keep = [((w >> (8 * b)) & 0xff) >= t for b in range(4)]
    half = lambda k: np.where(k, np.uint32(0xffff), np.uint32(0))
    want_lo = half(keep[0]) | (half(keep[1]) << np.uint32(16))
    want_hi = half(keep[2]) | (half(keep[3]) << np.uint32(16))
    assert np.array_equal(got[:, 0], want_lo) and np.array_equal(got[:, 1], want_hi)
    # the per-key 32-bit masks of the backward's dS step
    got = _run(probe, recs, mode=6)
    for b in range(4):
        assert np.array_equal(got[:, b], np.where(keep[b], np.uint32(0xffffffff), np.uint32(0)))
