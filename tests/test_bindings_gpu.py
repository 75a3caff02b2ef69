"""The Python binding's checks of caller-supplied output buffers: every
wrapper that takes `out` / `lse` refuses a tensor that does not hold exactly
what the C call writes (element count, dtype, device, contiguity), so a
wrong buffer raises ValueError instead of being written past."""
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


def _bad_buffers(shape, dtype):
    dev = torch.device("cuda")
    n = 1
    for d in shape:
        n *= d
    other = torch.float32 if dtype == torch.bfloat16 else torch.bfloat16
    return [torch.empty(n + 1, dtype=dtype, device=dev),
            torch.empty(shape, dtype=other, device=dev),
            torch.empty(shape, dtype=dtype),                                       # CPU
            torch.empty(tuple(shape[:-1]) + (2 * shape[-1],), dtype=dtype, device=dev)[..., ::2]]


def test_forward_and_dropout_reject_bad_outputs():
    q = torch.randn(1, 2, 130, 64, device="cuda").to(torch.bfloat16)
    for bad in _bad_buffers((1, 2, 130, 64), torch.bfloat16):
        with pytest.raises(ValueError):
            fa.forward(q, q, q, out=bad)
        with pytest.raises(ValueError):
            fa.forward_dropout(q, q, q, 0.1, 1, out=bad)
    for bad in _bad_buffers((1, 2, 130), torch.float32):
        with pytest.raises(ValueError):
            fa.forward(q, q, q, lse=bad)
        with pytest.raises(ValueError):
            fa.forward_dropout(q, q, q, 0.1, 1, lse=bad)
    # the right buffers, in another shape with the same elements, are taken
    o = torch.empty(2, 130, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(260, dtype=torch.float32, device="cuda")
    out, l2 = fa.forward(q, q, q, out=o, lse=lse)
    assert out is o and l2 is lse
    ref, lref = fa.forward(q, q, q)
    assert torch.equal(o.view_as(ref), ref) and torch.equal(lse.view_as(lref), lref)


def test_softmax_rejects_bad_outputs():
    x = torch.randn(33, 100, device="cuda")
    for bad in _bad_buffers((33, 100), torch.float32):
        with pytest.raises(ValueError):
            fa.softmax_rows(x, out=bad)
    for bad in _bad_buffers((33,), torch.float32):
        with pytest.raises(ValueError):
            fa.softmax_rows(x, lse=bad)


def test_decode_paged_rejects_bad_outputs():
    B, H, D, page, pages = 2, 2, 64, 16, 4
    q = torch.randn(B, H, D, device="cuda").to(torch.bfloat16)
    kc = torch.randn(pages, page, H, D, device="cuda").to(torch.bfloat16)
    bt = torch.arange(pages, dtype=torch.int32, device="cuda").view(B, 2)
    lens = torch.tensor([20, 32], dtype=torch.int32, device="cuda")
    for bad in _bad_buffers((B, H, D), torch.bfloat16):
        with pytest.raises(ValueError):
            fa.decode_paged(q, kc, kc, bt, lens, out=bad)
    for bad in _bad_buffers((B, H), torch.float32):
        with pytest.raises(ValueError):
            fa.decode_paged(q, kc, kc, bt, lens, lse=bad)
    with pytest.raises(ValueError):
        fa.decode_paged(q, kc, kc, bt.cpu(), lens)
