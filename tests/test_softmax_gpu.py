"""GPU parity of the two-read row softmax (fa_softmax_rows through the C ABI)
with the fp64 oracle oracle.softmax, element by element: short rows (one warp
per row), long rows read through shared memory (aligned, a multiple of 4
columns, up to 16384 of them; several rows per CTA through its two row
buffers) and the other long rows (one CTA per row from global memory),
column counts that are not a multiple of 4, unaligned input or output,
single-column rows, in place, masked (-inf) entries and all-masked rows,
large logits, and a 1 GiB matrix checked on sampled rows."""
import numpy as np
import pytest
import torch

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build
from oracle.softmax import softmax_rows as oracle_softmax

pytestmark = pytest.mark.gpu

# fp32 output in [0, 1]: ex2.approx (relative error ~2^-22) and fp32 sums
ATOL_Y = 2e-6
ATOL_LSE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa_build.build()
    fa.load()
    torch.cuda.init()


def _compare(x, y, lse, rows=None):
    xs = x.cpu().numpy() if rows is None else x[rows].cpu().numpy()
    ry, rl = oracle_softmax(xs)
    gy = (y if rows is None else y[rows]).cpu().numpy().astype(np.float64)
    gl = (lse if rows is None else lse[rows]).cpu().numpy().astype(np.float64)
    assert np.abs(gy - ry).max() <= ATOL_Y
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(gl), ~fin)
    if fin.any():
        assert np.abs(gl[fin] - rl[fin]).max() <= ATOL_LSE * max(1.0, np.abs(rl[fin]).max())


def _x(rows, cols, seed, std=3.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).cuda()


@pytest.mark.parametrize("cols", [1, 3, 4, 5, 127, 128, 2048, 2049, 2052, 3000, 16384, 16388, 65536])
def test_shapes(cols):
    rows = max(1, min(300, (1 << 22) // cols))
    x = _x(rows, cols, cols)
    y, lse = fa.softmax_rows(x)
    _compare(x, y, lse)


def test_in_place_and_large_logits():
    x = _x(64, 4096, 5, std=200.0)
    ref_y, ref_lse = fa.softmax_rows(x.clone())
    y, lse = fa.softmax_rows(x, out=x)
    assert torch.equal(y, ref_y) and torch.equal(lse, ref_lse)
    _compare(_x(64, 4096, 5, std=200.0), y, lse)


def test_masked_entries_and_empty_rows():
    x = _x(40, 1000, 6)
    x[:, ::3] = float("-inf")
    x[7] = float("-inf")
    x[30, :998] = float("-inf")            # column 999 is masked too (999 % 3 == 0)
    y, lse = fa.softmax_rows(x)
    _compare(x, y, lse)
    assert torch.all(y[7] == 0) and torch.isneginf(lse[7])
    assert y[30, 998].item() == 1.0


def test_one_gib_sampled_rows():
    x = _x(1, 1, 0)  # warm-up allocation
    g = torch.Generator(device="cuda").manual_seed(8)
    x = torch.randn(32768, 8192, generator=g, device="cuda") * 4
    y, lse = fa.softmax_rows(x)
    rows = torch.randperm(32768, generator=torch.Generator().manual_seed(9))[:64].sort().values
    _compare(x, y, lse, rows=rows.cuda())
    torch.testing.assert_close(y.double().sum(-1), torch.ones(32768, dtype=torch.float64, device="cuda"),
                               atol=1e-5, rtol=0)
    del x, y
    torch.cuda.empty_cache()


def test_shared_memory_rows_masked_and_many_rows_per_cta():
    # 2000 rows of 4096 on a few hundred CTAs: each CTA's two buffers cycle
    # through several phases; masked columns and an all-masked row
    x = _x(2000, 4096, 11)
    x[:, ::5] = float("-inf")
    x[17] = float("-inf")
    y, lse = fa.softmax_rows(x)
    _compare(x, y, lse)
    assert torch.all(y[17] == 0) and torch.isneginf(lse[17])


@pytest.mark.parametrize("shift_x,shift_y", [(1, 0), (0, 1), (2, 3)])
def test_unaligned_input_or_output(shift_x, shift_y):
    # views starting 4, 8 or 12 bytes into their storage: an unaligned input
    # takes the global-memory kernel, an unaligned output the scalar stores
    rows, cols = 300, 4096
    src = _x(rows, cols, 13)
    xb = torch.empty(rows * cols + 4, dtype=torch.float32, device="cuda")
    yb = torch.empty(rows * cols + 4, dtype=torch.float32, device="cuda")
    x = xb[shift_x:shift_x + rows * cols].view(rows, cols)
    x.copy_(src)
    y = yb[shift_y:shift_y + rows * cols].view(rows, cols)
    out, lse = fa.softmax_rows(x, out=y)
    _compare(src, out, lse)
    # the aligned call may take the other kernel, whose sums run in another
    # order: the two agree within the oracle bound
    ref, ref_lse = fa.softmax_rows(src)
    torch.testing.assert_close(out, ref, atol=ATOL_Y, rtol=0)
