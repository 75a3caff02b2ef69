"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, element by element, at small sizes spanning several
tiles and ragged tails, at the full workload sizes on sampled rows/heads, and
on edge cases (single key, single query, causal row 0, lengths that are not a
multiple of the 128-row tile)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from exact_attention_03_gb300.inputs import (SWEEP_LENGTHS, WORKLOADS, Workload, make_inputs,
                                             sample_rows)
from parity_util import ATOL_LSE, ATOL_O, assert_parity, compare_heads, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _dev(*ts):
    return [t.cuda() for t in ts]


# ---------------------------------------------------------------- workloads

def test_mha_l256_d64_full():
    w = WORKLOADS["mha_l256_d64"]
    q, k, v = _dev(*make_inputs(w, "cpu"))
    do, dl, n = assert_parity(q, k, v, w.causal)
    assert n == w.B * w.H * w.Lq


@pytest.mark.parametrize("L", SWEEP_LENGTHS)
def test_sweep_d64(L):
    w = WORKLOADS[f"sweep_d64_L{L}"]
    q, k, v = _dev(*make_inputs(w, "cpu"))
    if L <= 1024:
        assert_parity(q, k, v, w.causal)
    else:
        g = torch.Generator().manual_seed(L)
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
        rows = []
        for _ in heads:
            r = torch.randperm(L, generator=g)[:62]
            rows.append(torch.sort(torch.cat([torch.tensor([0, L - 1]), r])).values.numpy())
        assert_parity(q, k, v, w.causal, heads=heads, rows=rows)


def _boundary_rows(L, extra, seed):
    g = torch.Generator().manual_seed(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, L // 2, L - 129, L - 128, L - 2, L - 1]
    r = torch.randperm(L, generator=g)[:extra]
    return np.unique(np.clip(np.concatenate([np.array(fixed), r.numpy()]), 0, L - 1))


def test_causal_l8k_d128_sampled():
    w = WORKLOADS["causal_l8k_d128"]
    q, k, v = make_inputs(w, "cuda")
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    rows = [_boundary_rows(w.Lq, 36, 100 + i) for i in range(len(heads))]
    assert_parity(q, k, v, w.causal, heads=heads, rows=rows)


@pytest.mark.slow
def test_causal_l64k_d128_sampled_rows():
    w = WORKLOADS["causal_l64k_d128"]
    q, k, v = make_inputs(w, "cuda")
    heads = [(0, h) for h in range(w.H)]
    rows = [r.numpy() for r in sample_rows(w)]
    assert len(rows) == w.H and all(len(r) == 512 for r in rows)
    assert_parity(q, k, v, w.causal, heads=heads, rows=rows)


@pytest.mark.slow
def test_decode_l128k_d128_sampled_heads():
    w = WORKLOADS["decode_l128k_d128"]
    q, k, v = make_inputs(w, "cuda")
    g = torch.Generator().manual_seed(4 + 2000)
    flat = torch.randperm(w.B * w.H, generator=g)[:62].tolist() + [0, w.B * w.H - 1]
    heads = sorted({(i // w.H, i % w.H) for i in flat})
    o, lse = run_gpu(q, k, v, w.causal)
    torch.cuda.synchronize()
    do, dl, n = compare_heads(q, k, v, o, lse, w.scale, w.causal, heads=heads)
    assert do <= ATOL_O and dl <= ATOL_LSE, (do, dl)
    # every head: the output is a convex combination of the value rows
    vmin = v.float().amin(dim=2)
    vmax = v.float().amax(dim=2)
    of = o.float()[:, :, 0]
    assert bool(((of >= vmin - 1e-2) & (of <= vmax + 1e-2)).all())
    assert bool(torch.isfinite(lse).all())


# ---------------------------------------------------------------- edge cases

EDGE = [
    # B, H, Lq, Lk, D, causal
    (1, 1, 1, 1, 64, False),       # single key, single query (decode path)
    (1, 1, 1, 1, 128, True),       # causal L = 1 (prefill path)
    (1, 2, 5, 5, 64, True),
    (1, 1, 1, 7, 128, False),
    (2, 2, 1, 300, 128, False),
    (1, 3, 1, 4097, 64, False),
    (1, 1, 1, 50000, 128, False),
    (2, 3, 200, 200, 128, True),
    (1, 2, 300, 700, 64, False),
    (1, 2, 700, 300, 128, False),
    (1, 1, 129, 129, 128, False),
    (1, 1, 127, 255, 128, False),
    (3, 1, 384, 384, 64, True),
    (1, 1, 640, 640, 128, True),
    (1, 2, 2, 2000, 64, False),
    (1, 1, 1000, 1, 128, False),
    (2, 1, 513, 513, 64, True),
]


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", EDGE)
def test_edge_shapes(B, H, Lq, Lk, D, causal):
    w = Workload("edge", B, H, Lq, Lk, D, causal, seed=7)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    assert_parity(q, k, v, causal)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_sharp_logits(D, causal):
    # q, k drawn x3: logits with std ~9 exercise the rescale path on every tile
    w = Workload("sharp", 1, 4, 777, 777, D, causal, seed=9, qk_std=3.0)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    assert_parity(q, k, v, causal)


@pytest.mark.parametrize("D", [64, 128])
def test_late_outliers_force_rescale(D):
    # large keys placed only at the end of the sequence: the running max keeps
    # growing tile after tile
    w = Workload("late", 1, 2, 512, 1536, D, False, seed=11)
    q, k, v = make_inputs(w, "cpu")
    k = k.clone()
    k[:, :, 1024:] = (k[:, :, 1024:].float() * 6).to(torch.bfloat16)
    q, k, v = _dev(q, k, v)
    assert_parity(q, k, v, False)


@pytest.mark.parametrize("D", [64, 128])
def test_running_max_growth_per_tile(D):
    # scale = ln 2 makes the base-2 logit equal to q.k.  q = (1, 0.1 n): key
    # tile 0 scores ~0, tile 1 ~1.5 (its weights against the old maximum sum
    # past 2^8 although no weight grows past 2^8), tile 2 ~12 (a growth past
    # 2^8 after the first tile: rescale O and recompute the tile), tile 3
    # back to ~0, and a ragged tile 4.
    g = torch.Generator().manual_seed(21)
    B, H, Lq, Lk = 1, 2, 600, 600
    q = torch.randn(B, H, Lq, D, generator=g) * 0.1
    q[..., 0] = 1.0
    k = torch.randn(B, H, Lk, D, generator=g)
    k[..., 0] = 0.0
    k[:, :, 128:256, 0] = 1.5
    k[:, :, 256:384, 0] = 12.0
    v = torch.randn(B, H, Lk, D, generator=g)
    q, k, v = _dev(*(t.to(torch.bfloat16) for t in (q, k, v)))
    assert_parity(q, k, v, False, scale=math.log(2.0))
    assert_parity(q, k, v, True, scale=math.log(2.0))


def test_custom_scale():
    w = Workload("scale", 1, 2, 300, 300, 64, True, seed=12)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    assert_parity(q, k, v, True, scale=0.37)


def test_constant_values_return_the_value_row():
    w = Workload("const", 2, 2, 260, 260, 128, True, seed=13)
    q, k, v = make_inputs(w, "cpu")
    row = torch.randn(128).to(torch.bfloat16)
    v = row.expand_as(v).contiguous()
    q, k, v = _dev(q, k, v)
    o, lse = run_gpu(q, k, v, True)
    assert torch.allclose(o.float(), v.float(), atol=2e-2, rtol=0)


def test_deterministic_and_stream_ordered():
    w = Workload("det", 1, 4, 1000, 1000, 128, True, seed=14)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = run_gpu(q, k, v, True, stream=s)
        o2, l2 = run_gpu(q, k, v, True, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional():
    w = Workload("nolse", 1, 1, 256, 256, 64, False, seed=15)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    o_ref, _ = run_gpu(q, k, v, False)
    o, lse = fa.forward(q, k, v, return_lse=False)
    assert lse is None
    assert fa.last_device_error()[0] == fa.FA_OK
    assert torch.equal(o, o_ref)


def test_host_buffers_end_to_end():
    w = Workload("host", 1, 2, 333, 333, 128, True, seed=16)
    q, k, v = (t.pin_memory() for t in make_inputs(w, "cpu"))
    oh, lh = fa.forward_host(q, k, v, causal=True)
    assert not oh.is_cuda
    od, ld = run_gpu(q.cuda(), k.cuda(), v.cuda(), True)
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_gives_up_and_context_survives():
    """A barrier nothing completes: the bounded wait must return after its
    limit with FA_ERR_TIMEOUT, and the next attention call must still work."""
    assert fa.wait_selftest(20000) == fa.FA_ERR_TIMEOUT
    assert fa.last_device_error()[0] == fa.FA_OK  # the word was read and cleared
    w = Workload("after", 1, 1, 256, 256, 64, False, seed=17)
    q, k, v = _dev(*make_inputs(w, "cpu"))
    assert_parity(q, k, v, False)
