"""Host-side checks of the C ABI: the library loads, exports every function
include/fa.h declares, and rejects bad arguments before any CUDA call.
No kernel is launched here (bad arguments never reach the GPU)."""
import ctypes
import os
import re

import pytest

import exact_attention_03_gb300 as fa
from exact_attention_03_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_strerror", "fa_last_device_error", "fa_decode_num_splits",
              "fa_wait_selftest", "fa_abi_version", "fa_fwd_decode_paged", "fa_softmax_rows",
              "fa_bwd", "fa_bwd_dropout", "fa_fwd_dropout", "fa_fwd_host", "fa_host_num_chunks",
              "fa_fwd_host_async"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding knows the signature of each of them
    assert set(declared_functions()) <= set(fa.EXPORTED_SYMBOLS)


def test_abi_version(lib):
    assert lib.fa_abi_version() == (1 << 16) | 6


def test_strerror_covers_every_status(lib):
    for code in range(0, -6, -1):
        s = fa.strerror(code)
        assert s and "unknown" not in s
    assert "unknown" in fa.strerror(-99)


A = 0x10000  # a 16-byte aligned fake address; calls below never dereference it


def call(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Lq=128, Lk=128, D=128, scale=0.1, causal=0)
    args.update(kw)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                     args["Lq"], args["Lk"], args["D"], args["scale"], args["causal"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Lq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Lk=0), fa.FA_ERR_INVALID_ARG),
    (dict(D=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(D=256), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=1, Lq=64, Lk=128), fa.FA_ERR_UNSUPPORTED),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(k=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(v=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 1), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_bad_arguments_rejected_on_host(lib, kw, expect):
    assert call(**kw) == expect


def test_valid_arguments_without_a_gpu_report_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (the fake pointers must never reach a kernel)")
    assert call() == fa.FA_ERR_CUDA
    assert call(Lq=1, Lk=1000) == fa.FA_ERR_CUDA
    st, site = fa.last_device_error(None)
    assert st == fa.FA_ERR_CUDA and site == 0


@pytest.mark.parametrize("BH,Lk,sms", [(512, 131072, 152), (1, 131072, 152), (32, 256, 148),
                                       (1, 1, 152), (7, 65, 152), (4096, 100000, 152),
                                       (1, 10 ** 9, 152), (3, 4097, 1)])
def test_decode_split_count(lib, BH, Lk, sms):
    n = fa.decode_num_splits(BH, Lk, sms)
    assert 1 <= n <= 4096
    chunk = -(-Lk // n)
    assert (n - 1) * chunk < Lk, "no split may be empty"
    assert chunk >= min(64, Lk) or n == 1
    if (BH, Lk, sms) == (512, 131072, 152):
        assert n == 64  # 2048 keys per split
    assert fa.decode_num_splits(0, 10, 10) == fa.FA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "_HERE", str(tmp_path))
    with pytest.raises(ImportError):
        fa.load()


def test_wait_selftest_rejects_bad_limit(lib):
    assert fa.wait_selftest(0) == fa.FA_ERR_INVALID_ARG
    assert fa.wait_selftest(10 ** 8) == fa.FA_ERR_INVALID_ARG


def test_binding_rejects_bad_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)  # CPU tensors are refused; no silent fallback
    with pytest.raises(ValueError):
        fa.forward(q[0], q, q)
    lse = torch.zeros(1, 1, 4)
    with pytest.raises(ValueError):
        fa.backward(q, q, q, q, lse, q)
    with pytest.raises(ValueError):
        fa.backward_dropout(q, q, q, q, lse, q, 0.1, 1)
    with pytest.raises(ValueError):
        fa.backward(q[0], q, q, q, lse, q)
    # caller-supplied host outputs must hold what the call writes
    for kw in (dict(out=torch.empty(1, 1, 3, 64, dtype=torch.bfloat16)),
               dict(out=torch.empty(1, 1, 4, 64, dtype=torch.float32)),
               dict(out=torch.empty(1, 1, 64, 4, dtype=torch.bfloat16).transpose(2, 3)),
               dict(lse=torch.empty(1, 1, 5)),
               dict(lse=torch.empty(1, 1, 4, dtype=torch.float64))):
        with pytest.raises(ValueError):
            fa.forward_host(q, q, q, **kw)


def call_paged(**kw):
    args = dict(q=A, kc=A, vc=A, bt=A, lens=A, o=A, lse=A, B=2, H=4, D=128, num_pages=64,
                page_size=16, max_pages=8, scale=0.1)
    args.update(kw)
    return fa.load().fa_fwd_decode_paged(args["q"], args["kc"], args["vc"], args["bt"], args["lens"],
                                         args["o"], args["lse"], args["B"], args["H"], args["D"],
                                         args["num_pages"], args["page_size"], args["max_pages"],
                                         args["scale"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(kc=None), fa.FA_ERR_INVALID_ARG),
    (dict(vc=None), fa.FA_ERR_INVALID_ARG),
    (dict(bt=None), fa.FA_ERR_INVALID_ARG),
    (dict(lens=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=0), fa.FA_ERR_INVALID_ARG),
    (dict(num_pages=0), fa.FA_ERR_INVALID_ARG),
    (dict(page_size=0), fa.FA_ERR_INVALID_ARG),
    (dict(page_size=24), fa.FA_ERR_INVALID_ARG),
    (dict(page_size=1 << 17), fa.FA_ERR_INVALID_ARG),
    (dict(max_pages=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(page_size=1 << 16, max_pages=1 << 16), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(kc=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(vc=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(bt=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(lens=A + 1), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_paged_bad_arguments_rejected_on_host(lib, kw, expect):
    assert call_paged(**kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(x=None), fa.FA_ERR_INVALID_ARG),
    (dict(y=None), fa.FA_ERR_INVALID_ARG),
    (dict(rows=0), fa.FA_ERR_INVALID_ARG),
    (dict(cols=0), fa.FA_ERR_INVALID_ARG),
    (dict(rows=1 << 40, cols=2), fa.FA_ERR_UNSUPPORTED),
    (dict(x=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(y=A + 1), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_softmax_bad_arguments_rejected_on_host(lib, kw, expect):
    args = dict(x=A, y=A, lse=A, rows=4, cols=16)
    args.update(kw)
    assert lib.fa_softmax_rows(args["x"], args["y"], args["lse"], args["rows"], args["cols"], None) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(do=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(dq=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Lk=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=1, Lq=64, Lk=128), fa.FA_ERR_UNSUPPORTED),
    (dict(o=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(dk=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_bwd_bad_arguments_rejected_on_host(lib, kw, expect):
    a = dict(q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, Lq=128, Lk=128, D=128,
             scale=0.1, causal=0)
    a.update(kw)
    assert lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"],
                      a["B"], a["H"], a["Lq"], a["Lk"], a["D"], a["scale"], a["causal"], None) == expect


BWD_DROPOUT_CASES = [
    (dict(p=-0.1), fa.FA_ERR_INVALID_ARG),
    (dict(p=1.0), fa.FA_ERR_INVALID_ARG),
    (dict(p=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(p=0.999), fa.FA_ERR_INVALID_ARG),      # rounds to 256/256
]


@pytest.mark.parametrize("kw,expect", BWD_DROPOUT_CASES + [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(dv=None), fa.FA_ERR_INVALID_ARG),
    (dict(H=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(causal=-1), fa.FA_ERR_INVALID_ARG),
    (dict(D=32), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=1, Lq=128, Lk=256), fa.FA_ERR_UNSUPPORTED),
    (dict(do=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_bwd_dropout_bad_arguments_rejected_on_host(lib, kw, expect):
    a = dict(q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, Lq=128, Lk=128, D=64,
             scale=0.1, causal=0, p=0.1, seed=(1 << 64) - 1, offset=(1 << 32) - 1)
    a.update(kw)
    assert lib.fa_bwd_dropout(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"],
                              a["B"], a["H"], a["Lq"], a["Lk"], a["D"], a["scale"], a["causal"], a["p"],
                              a["seed"], a["offset"], None) == expect


def test_bwd_dropout_valid_arguments_without_a_gpu_report_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (the fake pointers must never reach a kernel)")
    assert lib.fa_bwd_dropout(A, A, A, A, A, A, A, A, A, 1, 1, 128, 128, 128, 0.1, 1, 0.5, 3, 7,
                              None) == fa.FA_ERR_CUDA


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(p=-0.1), fa.FA_ERR_INVALID_ARG),
    (dict(p=1.0), fa.FA_ERR_INVALID_ARG),
    (dict(p=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(p=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(p=0.999), fa.FA_ERR_INVALID_ARG),      # rounds to 256/256
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=1, Lq=64, Lk=128), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_dropout_bad_arguments_rejected_on_host(lib, kw, expect):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Lq=128, Lk=128, D=128, scale=0.1, causal=0, p=0.1,
             seed=1, offset=0)
    a.update(kw)
    assert lib.fa_fwd_dropout(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Lq"], a["Lk"],
                              a["D"], a["scale"], a["causal"], a["p"], a["seed"], a["offset"], None) == expect


def test_dropout_valid_arguments_without_a_gpu_report_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (the fake pointers must never reach a kernel)")
    assert lib.fa_fwd_dropout(A, A, A, A, A, 1, 1, 128, 128, 64, 0.1, 0, 0.998, (1 << 64) - 1, 7, None) == fa.FA_ERR_CUDA


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(H=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(causal=5), fa.FA_ERR_INVALID_ARG),
    (dict(D=80), fa.FA_ERR_UNSUPPORTED),
    (dict(causal=1, Lq=64, Lk=128), fa.FA_ERR_UNSUPPORTED),
])
def test_host_entry_bad_arguments_rejected_on_host(lib, kw, expect):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Lq=128, Lk=128, D=128, scale=0.1, causal=0)
    a.update(kw)
    assert lib.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Lq"], a["Lk"], a["D"],
                           a["scale"], a["causal"], None) == expect


@pytest.mark.parametrize("BH,per,expect", [(1, 1, 1), (2, 300 * 128 * 8, 1), (32, 8192 * 64 * 8, 8),
                                           (13, 2048 * 128 * 8, 3), (3, 1 << 30, 3), (1000, 1 << 20, 8),
                                           (17, 1 << 22, 6), (0, 5, 1), (5, 0, 1)])
def test_host_chunk_rule(lib, BH, per, expect):
    # min(8, BH, BH * per / 8 MiB) chunks, at least 1, then as many as equal head counts need
    n = lib.fa_host_num_chunks(BH, per)
    assert n == expect
    if BH > 0 and per > 0:
        hc = -(-BH // n)
        assert (n - 1) * hc < BH <= n * hc


def test_host_async_entry_rejects_bad_arguments_on_host(lib):
    assert lib.fa_fwd_host_async(None, A, A, A, A, 1, 1, 128, 128, 128, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_host_async(A, A, A, A, A, 1, 1, 128, 128, 96, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED
