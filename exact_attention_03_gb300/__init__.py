"""GB300 (sm_103a) exact-attention forward: thin Python binding of libfa_gb300.so.

Every step of the computation runs in the library's CUDA kernels; this module
only marshals arguments (pointers, sizes, the current CUDA stream) through the
C ABI declared in include/fa.h.  PyTorch is used for device memory and
streams.  There is no fallback: if the library is missing, or the call fails,
an exception is raised.

    import exact_attention_03_gb300 as fa
    o, lse = fa.forward(q, k, v, causal=True)          # bf16 [B,H,L,D] on cuda
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

__all__ = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
           "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FlashAttentionError", "lib_path", "load",
           "fa_fwd", "strerror", "last_device_error", "wait_selftest", "decode_num_splits",
           "forward", "forward_host", "decode_noalloc", "decode_paged", "softmax_rows",
           "backward", "backward_dropout", "forward_dropout", "EXPORTED_SYMBOLS"]

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_MISALIGNED = -3
FA_ERR_CUDA = -4
FA_ERR_TIMEOUT = -5

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libfa_gb300.so"
_lib = None

# name -> (restype, argtypes)
_SIGS = {
    "fa_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                              ctypes.c_void_p]),
    "fa_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_last_device_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]),
    "fa_decode_num_splits": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "fa_wait_selftest": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p]),
    "fa_abi_version": (ctypes.c_int, []),
    "fa_fwd_decode_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_float, ctypes.c_void_p]),
    "fa_decode_noalloc_max_floats": (ctypes.c_int, []),
    "fa_fwd_decode_paged": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_float, ctypes.c_void_p]),
    "fa_softmax_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p]),
    "fa_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5
               + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_dropout": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                       + [ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong,
                          ctypes.c_uint, ctypes.c_void_p]),
    "fa_bwd_dropout": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5
                       + [ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong,
                          ctypes.c_uint, ctypes.c_void_p]),
    "fa_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                    + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "fa_host_num_chunks": (ctypes.c_int, [ctypes.c_longlong, ctypes.c_longlong]),
    "fa_fwd_host_async": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                          + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)


class FlashAttentionError(RuntimeError):
    def __init__(self, status: int, what: str = "fa_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {status} ({strerror(status)})")


def lib_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load():
    """Loads the CUDA library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with exact_attention_03_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    try:
        return load().fa_strerror(int(status)).decode()
    except ImportError:
        return f"status {status}"


def fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Lq, Lk, D, scale, causal, stream) -> int:
    """Raw C-ABI call: integer pointers / sizes in, status code out."""
    return load().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Lq, Lk, D,
                         float(scale), int(causal), stream)


def last_device_error(stream=None) -> Tuple[int, int]:
    """(status, wait site) of the device error word; synchronises `stream`."""
    site = ctypes.c_int(0)
    st = load().fa_last_device_error(_stream_handle(stream), ctypes.byref(site))
    return st, site.value


def wait_selftest(limit_us: int = 20000, stream=None) -> int:
    return load().fa_wait_selftest(int(limit_us), _stream_handle(stream))


def decode_num_splits(BH: int, Lk: int, num_sms: int) -> int:
    return load().fa_decode_num_splits(int(BH), int(Lk), int(num_sms))


def _check_out(name, t, numel, dtype, device):
    """A caller-supplied output tensor: the C call writes `numel` elements of
    `dtype` to its data pointer, so it must hold exactly that many,
    contiguously, on `device` (a torch.device, or "cpu" for host buffers)."""
    on_device = (not t.is_cuda) if device == "cpu" else (t.is_cuda and t.device == device)
    if t.numel() != numel or t.dtype != dtype or not t.is_contiguous() or not on_device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of {numel} elements on {device}")


def _stream_handle(stream):
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return stream


def forward(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None,
            lse=None, return_lse: bool = True, stream=None):
    """O (bf16 [B,H,Lq,D]) and LSE (fp32 [B,H,Lq]) for CUDA bf16 q [B,H,Lq,D],
    k, v [B,H,Lk,D].  `scale` defaults to 1/sqrt(D)."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, H, Lq, D = q.shape
    if k.shape != (B, H, k.shape[2], D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA bf16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, H, Lq, D), dtype=torch.bfloat16, device=q.device)
    else:
        _check_out("out", out, B * H * Lq * D, torch.bfloat16, q.device)
    if return_lse and lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _check_out("lse", lse, B * H * Lq, torch.float32, q.device)
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, H, Lq, Lk, D, scale,
                int(causal), _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st)
    return out, lse


def forward_dropout(q, k, v, p_drop: float, seed: int, offset: int = 0, causal: bool = False,
                    scale: Optional[float] = None, out=None, lse=None, stream=None):
    """forward() with dropout on the attention weights, fused into the kernel
    (fa_fwd_dropout): weights are kept iff their Philox byte >= round(256 p),
    kept ones scaled by 256 / (256 - round(256 p)); lse is the undropped
    log-sum-exp.  `seed` (64-bit) and `offset` (32-bit) select the bits."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, H, Lq, D = q.shape
    if k.shape != (B, H, k.shape[2], D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA bf16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, H, Lq, D), dtype=torch.bfloat16, device=q.device)
    else:
        _check_out("out", out, B * H * Lq * D, torch.bfloat16, q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    else:
        _check_out("lse", lse, B * H * Lq, torch.float32, q.device)
    st = load().fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, H, Lq, Lk, D, scale, int(causal), float(p_drop),
                               int(seed) & ((1 << 64) - 1), int(offset) & 0xFFFFFFFF,
                               _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, "fa_fwd_dropout")
    return out, lse


def decode_noalloc(q, k, v, scale: Optional[float] = None, out=None, lse=None, stream=None):
    """Single-query attention (q [B,H,1,D], k, v [B,H,Lk,D]) through
    fa_fwd_decode_noalloc, which uses the library's fixed device array instead
    of allocating a workspace (for callers that must not allocate while they
    run).  Pass `out` (bf16 [B,H,1,D]) and `lse` (fp32 [B,H,1]) for a call
    that allocates nothing at all: when omitted, this wrapper creates them
    with torch.  The caller must not run two such calls concurrently on the
    GPU."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, H, Lq, D = q.shape
    if Lq != 1:
        raise ValueError("decode_noalloc takes one query row per head")
    if k.shape != (B, H, k.shape[2], D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, H, 1, D), dtype=torch.bfloat16, device=q.device)
    elif (tuple(out.shape) != (B, H, 1, D) or out.dtype != torch.bfloat16 or out.device != q.device
          or not out.is_contiguous()):
        raise ValueError(f"out must be a contiguous bf16 tensor [B, H, 1, D] on {q.device}")
    if lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    elif (lse.numel() != B * H or lse.dtype != torch.float32 or lse.device != q.device
          or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous fp32 tensor of B*H elements on {q.device}")
    st = load().fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, H, Lk, D, float(scale),
                                      _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, "fa_fwd_decode_noalloc")
    return out, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale: Optional[float] = None,
                 out=None, lse=None, stream=None):
    """Single-query attention against a paged cache through fa_fwd_decode_paged.

    q: bf16 [B, H, D] or [B, H, 1, D]; k_cache, v_cache: bf16 [num_pages,
    page_size, H, D]; block_table: int32 [B, max_pages_per_seq]; seq_lens:
    int32 [B]; all CUDA tensors.  Returns O (bf16, shaped like q) and LSE
    (fp32 [B, H])."""
    import torch

    if q.dim() == 4:
        if q.shape[2] != 1:
            raise ValueError("decode_paged takes one query row per head")
        B, H, _, D = q.shape
    elif q.dim() == 3:
        B, H, D = q.shape
    else:
        raise ValueError("q must be [B, H, D] or [B, H, 1, D]")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache, v_cache must both be [num_pages, page_size, H, D]")
    num_pages, page_size, Hc, Dc = k_cache.shape
    if (Hc, Dc) != (H, D):
        raise ValueError(f"cache heads/dim {Hc, Dc} do not match q {H, D}")
    if block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages_per_seq] and seq_lens [B]")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor")
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    else:
        _check_out("out", out, B * H * D, torch.bfloat16, q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    else:
        _check_out("lse", lse, B * H, torch.float32, q.device)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("block_table", block_table),
                    ("seq_lens", seq_lens)):
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    st = load().fa_fwd_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, D, num_pages, page_size,
                                    block_table.shape[1], float(scale), _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, "fa_fwd_decode_paged")
    return out, lse


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None,
             dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv) of <dout, O> through fa_bwd, for CUDA bf16
    q, o, dout [B, H, Lq, D], k, v [B, H, Lk, D] and fp32 lse [B, H, Lq] from
    forward() with the same causal flag and scale."""
    return _backward(q, k, v, o, lse, dout, causal, scale, dq, dk, dv, stream, None)


def backward_dropout(q, k, v, o, lse, dout, p_drop: float, seed: int, offset: int = 0,
                     causal: bool = False, scale: Optional[float] = None, dq=None, dk=None,
                     dv=None, stream=None):
    """backward() for forward_dropout() (fa_bwd_dropout): o and lse are
    forward_dropout's outputs, and p_drop, seed and offset the ones it was
    called with; the kernels draw the same keep bits again."""
    return _backward(q, k, v, o, lse, dout, causal, scale, dq, dk, dv, stream,
                     (float(p_drop), int(seed) & ((1 << 64) - 1), int(offset) & 0xFFFFFFFF))


def _backward(q, k, v, o, lse, dout, causal, scale, dq, dk, dv, stream, drop):
    import torch

    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be [B, H, L, D]")
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, shape in (("q", q, (B, H, Lq, D)), ("k", k, (B, H, Lk, D)), ("v", v, (B, H, Lk, D)),
                           ("o", o, (B, H, Lq, D)), ("dout", dout, (B, H, Lq, D)),
                           ("dq", dq, (B, H, Lq, D)), ("dk", dk, (B, H, Lk, D)), ("dv", dv, (B, H, Lk, D))):
        if tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor of shape {shape}")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    if (tuple(lse.shape) != (B, H, Lq) or lse.dtype != torch.float32 or lse.device != q.device
            or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous fp32 tensor [B, H, Lq] on {q.device}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Lq, Lk, D,
            float(scale), int(causal))
    if drop is None:
        name = "fa_bwd"
        st = load().fa_bwd(*ptrs, _stream_handle(stream))
    else:
        name = "fa_bwd_dropout"
        st = load().fa_bwd_dropout(*ptrs, *drop, _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, name)
    return dq, dk, dv


def softmax_rows(x, out=None, lse=None, return_lse: bool = True, stream=None):
    """Row softmax of a CUDA fp32 tensor (last dimension = columns) through
    fa_softmax_rows.  Returns (y, lse) with y shaped like x and lse like
    x.shape[:-1] (None when return_lse is false)."""
    import torch

    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be a contiguous CUDA fp32 tensor")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols > 0 else 0
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_out("out", out, x.numel(), torch.float32, x.device)
    if return_lse and lse is None:
        lse = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    elif lse is not None:
        _check_out("lse", lse, rows, torch.float32, x.device)
    st = load().fa_softmax_rows(x.data_ptr(), out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, rows, cols,
                                _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, "fa_softmax_rows")
    return out, lse


def forward_host(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None, lse=None,
                 stream=None, sync: bool = True):
    """End-to-end call on host tensors through fa_fwd_host: q, k, v are CPU
    bf16 [B,H,L,D] tensors (page-locked for full copy bandwidth), O and LSE
    come back in page-locked CPU tensors.  The library pipelines the copies
    with the computation over chunks of heads.  With sync (the default) the
    call returns once the outputs are on the host; with sync=False it returns
    once the work is queued (fa_fwd_host_async) and the outputs are ready when
    `stream` (default: the current stream) has been synchronised."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, H, Lq, D = q.shape
    if k.shape != (B, H, k.shape[2], D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.is_cuda:
            raise ValueError(f"{name} must be a CPU bf16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is not None:
        _check_out("out", out, B * H * Lq * D, torch.bfloat16, "cpu")
    if lse is not None:
        _check_out("lse", lse, B * H * Lq, torch.float32, "cpu")
    if out is None:
        out = torch.empty((B, H, Lq, D), dtype=torch.bfloat16, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, pin_memory=True)
    fn = load().fa_fwd_host if sync else load().fa_fwd_host_async
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            B, H, Lq, Lk, D, scale, int(causal), _stream_handle(stream))
    if st != FA_OK:
        raise FlashAttentionError(st, "fa_fwd_host" if sync else "fa_fwd_host_async")
    return out, lse
