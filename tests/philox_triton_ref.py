"""Philox-4x32-10 words from Triton's library implementation, run on the CPU.

Test helper: an independent implementation of the generator (Triton's
``triton.language.random.philox_impl``, written by other authors from the
same published definition) against which the oracle's Philox is checked.
Triton's CPU interpreter must be switched on before Triton is imported, so
this runs as a child process:

    python tests/philox_triton_ref.py < request.json > words.json

request: {"ctr": [[c0, c1, c2, c3], ...], "key": [[k0, k1], ...]} (one key per
counter, each word below 2**32); reply: {"words": [[x0, x1, x2, x3], ...]}.
"""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402
from triton.language.random import philox_impl  # noqa: E402


@triton.jit
def _philox_kernel(inp, out, N: tl.constexpr):
    i = tl.arange(0, N)
    w = [tl.load(inp + 6 * i + c).to(tl.uint32, bitcast=True) for c in range(6)]
    x0, x1, x2, x3 = philox_impl(w[0], w[1], w[2], w[3], w[4], w[5], 10)
    tl.store(out + 4 * i + 0, x0.to(tl.int32, bitcast=True))
    tl.store(out + 4 * i + 1, x1.to(tl.int32, bitcast=True))
    tl.store(out + 4 * i + 2, x2.to(tl.int32, bitcast=True))
    tl.store(out + 4 * i + 3, x3.to(tl.int32, bitcast=True))


def words(ctr, key):
    n = len(ctr)
    N = 1
    while N < n:
        N *= 2
    flat = []
    for c, k in zip(ctr, key):
        flat.extend(list(c) + list(k))
    flat.extend([0] * 6 * (N - n))
    as_i32 = [v - (1 << 32) if v >= (1 << 31) else v for v in flat]
    inp = torch.tensor(as_i32, dtype=torch.int32)
    out = torch.zeros(4 * N, dtype=torch.int32)
    _philox_kernel[(1,)](inp, out, N)
    res = [v & 0xFFFFFFFF for v in out.tolist()]
    return [res[4 * r:4 * r + 4] for r in range(n)]


if __name__ == "__main__":
    req = json.load(sys.stdin)
    json.dump({"triton": triton.__version__, "words": words(req["ctr"], req["key"])}, sys.stdout)
