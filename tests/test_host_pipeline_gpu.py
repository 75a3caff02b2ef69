"""The host-buffer entry point fa_fwd_host pipelines copies and kernels over
chunks of heads; each head is computed by the same kernels as fa_fwd, so its
outputs must equal fa_fwd's on device copies of the same inputs bit for bit,
for every chunk count (1 .. 8), ragged last chunks, D 64/128, causal or not,
pageable and page-locked host memory and lse = NULL (the single-query path
splits the keys by the heads of one launch, so there only the last bits may
differ);
calls on another stream and repeated calls reuse the pipeline."""
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _host_inputs(B, H, Lq, Lk, D, seed, pinned=True):
    g = torch.Generator().manual_seed(seed)
    mk = lambda L: torch.randn(B, H, L, D, generator=g).to(torch.bfloat16)
    t = [mk(Lq), mk(Lk), mk(Lk)]
    return [x.pin_memory() for x in t] if pinned else t


def _chunks(B, H, Lq, Lk, D):
    return fa.load().fa_host_num_chunks(B * H, 2 * Lq * D * 2 + 2 * Lk * D * 2 + Lq * 4)


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [
    (1, 2, 300, 300, 128, True),          # one chunk (small)
    (2, 8, 4096, 4096, 64, False),        # 16 heads of 2 MiB: 4 chunks
    (1, 13, 2048, 2048, 128, True),       # ragged last chunk
    (4, 8, 8192, 8192, 64, False),        # the sweep's 8K length: 8 chunks
    (3, 5, 1, 40000, 128, False),         # single query rows (split-K/V kernels)
    (1, 3, 700, 1500, 64, False),         # Lq != Lk
])
def test_equals_device_forward(B, H, Lq, Lk, D, causal):
    q, k, v = _host_inputs(B, H, Lq, Lk, D, seed=B * 100 + H + Lq)
    n = _chunks(B, H, Lq, Lk, D)
    assert 1 <= n <= min(8, B * H)
    oh, lh = fa.forward_host(q, k, v, causal=causal)
    od, ld = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    assert fa.last_device_error()[0] == fa.FA_OK
    assert not oh.is_cuda and not lh.is_cuda
    if Lq == 1:
        # the single-query path picks its split count from the heads of one
        # launch, so the chunking changes its summation order: last bits only
        assert float((oh.float() - od.cpu().float()).abs().max()) <= 4e-3, f"{n} chunks"
        assert float((lh - ld.cpu()).abs().max()) <= 1e-5, f"{n} chunks"
    else:
        assert torch.equal(oh, od.cpu()), f"{n} chunks"
        assert torch.equal(lh, ld.cpu()), f"{n} chunks"


def test_chunk_counts_cover_one_to_eight():
    lib = fa.load()
    assert lib.fa_host_num_chunks(2, 300 * 128 * 8) == 1
    assert lib.fa_host_num_chunks(32, 8192 * 64 * 8) == 8
    assert lib.fa_host_num_chunks(13, 2048 * 128 * 8) == 3      # 26 MiB: 3 chunks of 5, 5, 3 heads
    assert lib.fa_host_num_chunks(3, 1 << 30) == 3               # never more chunks than heads


def test_pageable_memory_other_stream_and_no_lse():
    q, k, v = _host_inputs(1, 6, 1024, 1024, 128, seed=5, pinned=False)
    s = torch.cuda.Stream()
    oh, lh = fa.forward_host(q, k, v, causal=True, stream=s)
    od, ld = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())
    # lse = NULL through the C ABI
    o2 = torch.empty_like(q).pin_memory()
    st = fa.load().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), None, 1, 6, 1024, 1024,
                               128, 128 ** -0.5, 1, None)
    assert st == fa.FA_OK
    assert torch.equal(o2, od.cpu())


def test_repeated_calls_reuse_the_pipeline():
    q, k, v = _host_inputs(2, 8, 2048, 2048, 64, seed=9)
    outs = [fa.forward_host(q, k, v)[0].clone() for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_async_calls_queued_back_to_back():
    """Several problems queued with sync=False and one synchronisation: each
    output equals the device forward of its own inputs."""
    shapes = [(2, 8, 2048, 2048, 64, False), (1, 4, 1000, 1000, 128, True), (4, 8, 4096, 4096, 64, False),
              (1, 2, 1, 5000, 128, False)]
    probs = [(_host_inputs(*sh[:5], seed=20 + i), sh) for i, sh in enumerate(shapes)]
    outs = [fa.forward_host(q, k, v, causal=sh[5], sync=False) for (q, k, v), sh in probs]
    torch.cuda.current_stream().synchronize()
    for ((q, k, v), sh), (oh, lh) in zip(probs, outs):
        od, ld = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=sh[5])
        if sh[2] == 1:
            assert float((oh.float() - od.cpu().float()).abs().max()) <= 4e-3
            assert float((lh - ld.cpu()).abs().max()) <= 1e-5
        else:
            assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())
