"""Python binding of the GB300 NVFP4 quantizer C ABI (include/nvfp4.h).

Argument marshalling only: every step of the quantizer runs in the CUDA
library ``_build/libnvfp4.so`` (built by :func:`build`).  torch supplies device
memory and streams.  There is no CPU fallback: if the library is missing the
functions raise.

The functions keep the C names:

* :func:`nvfp4_amax`       -- float32[2] tensor amax (rowwise copy, columnwise copy)
* :func:`nvfp4_quantize`   -- packed E2M1 codes + E4M3 scales (+ alpha) per copy
* :func:`nvfp4_dequantize` -- codes + scales + alpha -> float32 or bfloat16
* :func:`nvfp4_gemm`       -- D = alpha_a * alpha_b * A * B^T of two NVFP4 operands (tiled scales)
* :func:`nvfp4_strerror`
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

from .build import LIB as _LIB_PATH
from .build import build

__all__ = [
    "ROWWISE", "COLWISE", "TWO_D", "RHT_ROW", "RHT_COL", "SR", "FOUR_SIX",
    "SEL_MAE", "SEL_MSE", "SEL_MAXERR", "Nvfp4Error", "Quantized", "lib", "build",
    "nvfp4_amax", "nvfp4_quantize", "nvfp4_dequantize", "nvfp4_gemm", "nvfp4_strerror", "output_shapes",
]

ROWWISE, COLWISE, TWO_D, RHT_ROW, RHT_COL, SR, FOUR_SIX, SF_SWIZZLED = 1, 2, 4, 8, 16, 32, 64, 128
SEL_MAE, SEL_MSE, SEL_MAXERR = 0, 1, 2

_lib: Optional[ctypes.CDLL] = None


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {nvfp4_strerror(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"NVFP4 CUDA library not built ({_LIB_PATH}); call "
                               "nvfp4_bit_block_gb300.build() first")
        L = ctypes.CDLL(_LIB_PATH)
        c = ctypes
        L.nvfp4_amax.restype = c.c_int
        L.nvfp4_amax.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_uint32, c.c_uint64,
                                 c.c_void_p, c.c_void_p]
        L.nvfp4_quantize.restype = c.c_int
        L.nvfp4_quantize.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p, c.c_uint32,
                                     c.c_int, c.c_uint64, c.c_uint64, c.c_uint64, c.c_void_p, c.c_void_p,
                                     c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p]
        L.nvfp4_dequantize.restype = c.c_int
        L.nvfp4_dequantize.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int64, c.c_int,
                                       c.c_void_p, c.c_void_p]
        L.nvfp4_error_histogram.restype = c.c_int
        L.nvfp4_error_histogram.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p, c.c_void_p,
                                            c.c_void_p, c.c_int, c.c_void_p, c.c_void_p]
        L.nvfp4_gemm.restype = c.c_int
        L.nvfp4_gemm.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
                                 c.c_int64, c.c_int64, c.c_int64, c.c_int, c.c_void_p, c.c_int64, c.c_void_p,
                                 c.c_void_p]
        L.nvfp4_strerror.restype = c.c_char_p
        L.nvfp4_strerror.argtypes = [c.c_int]
        _lib = L
    return _lib


def nvfp4_strerror(status: int) -> str:
    return lib().nvfp4_strerror(status).decode()


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise Nvfp4Error(status, where)


def _on_device(device, **tensors) -> None:
    """Every given tensor (None = absent) must live on `device`, a CUDA device:
    the kernels dereference these pointers on that GPU."""
    for name, t in tensors.items():
        if t is not None and (not t.is_cuda or t.device != device):
            raise ValueError(f"{name} must be a CUDA tensor on {device} (got {t.device})")


def _outs(q):
    return dict(q_row=q.q_row, s_row=q.s_row, q_col=q.q_col, s_col=q.s_col, alpha=q.alpha, status=q.status)


def _matrix(x):
    """(data_ptr, M, N, ld) of a 2-D bfloat16 CUDA tensor with unit column stride."""
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("x must be a 2-D torch.bfloat16 tensor")
    if not x.is_cuda:
        raise ValueError(f"x must be a CUDA tensor (got {x.device})")
    if x.size(1) > 0 and x.stride(1) != 1:
        raise ValueError("x must have unit stride along columns")
    ld = x.stride(0) if x.size(0) > 1 else max(x.size(1), 8)
    return x.data_ptr(), x.size(0), x.size(1), ld


def _scale_shape(rows: int, cols: int, swizzled: bool):
    """rows x cols scales; in the tiled layout rows pad to 128 and cols to 4."""
    if not swizzled:
        return (rows, cols)
    return (-(-rows // 128) * 128, -(-cols // 4) * 4)


def output_shapes(M: int, N: int, flags: int):
    """Shapes of (q_row, s_row, q_col, s_col) for an M x N tensor (None = not produced).
    With SF_SWIZZLED a scale buffer holds the padded tiled layout (its bytes
    are not a row-major matrix)."""
    row = bool(flags & ROWWISE)
    col = bool(flags & COLWISE)
    swz = bool(flags & SF_SWIZZLED)
    return ((M, N // 2) if row else None, _scale_shape(M, N // 16, swz) if row else None,
            (N, M // 2) if col else None, _scale_shape(N, M // 16, swz) if col else None)


@dataclass
class Quantized:
    q_row: object
    s_row: object
    q_col: object
    s_col: object
    alpha: object   # float32[2] device tensor
    status: object  # int32[1] device tensor (0, or NVFP4_ERR_NONFINITE / NVFP4_ERR_RANGE)


def nvfp4_amax(x, flags: int, rht_seed: int = 0, out=None, stream=None):
    """float32[2] device tensor: amax of the rowwise and the columnwise copy."""
    import torch
    p, M, N, ld = _matrix(x)
    if out is None:
        out = torch.empty(2, dtype=torch.float32, device=x.device)
    _on_device(x.device, out=out)
    with torch.cuda.device(x.device):
        _check(lib().nvfp4_amax(p, M, N, ld, flags, rht_seed, _ptr(out), _stream_handle(stream)),
               "nvfp4_amax")
    return out


def nvfp4_quantize(x, amax, flags: int, sel: int = SEL_MAE, sr_seed: int = 0, rht_seed: int = 0,
                   counter_offset: int = 0, out: Optional[Quantized] = None, stream=None) -> Quantized:
    """Quantize x (M x N bf16, CUDA) with the amax from :func:`nvfp4_amax`."""
    import torch
    p, M, N, ld = _matrix(x)
    if out is None:
        shapes = output_shapes(M, N, flags)
        mk = lambda s: None if s is None else torch.empty(s, dtype=torch.uint8, device=x.device)
        mks = mk if not flags & SF_SWIZZLED else (  # tiled scales: padding entries zero
            lambda s: None if s is None else torch.zeros(s, dtype=torch.uint8, device=x.device))
        q_row, s_row, q_col, s_col = shapes
        out = Quantized(mk(q_row), mks(s_row), mk(q_col), mks(s_col),
                        alpha=torch.empty(2, dtype=torch.float32, device=x.device),
                        status=torch.zeros(1, dtype=torch.int32, device=x.device))
    _on_device(x.device, amax=amax, **_outs(out))
    with torch.cuda.device(x.device):
        _check(lib().nvfp4_quantize(p, M, N, ld, _ptr(amax), flags, sel, sr_seed, rht_seed, counter_offset,
                                    _ptr(out.q_row), _ptr(out.s_row), _ptr(out.q_col), _ptr(out.s_col),
                                    _ptr(out.alpha), _ptr(out.status), _stream_handle(stream)),
               "nvfp4_quantize")
    return out


def nvfp4_dequantize(q, s, alpha, out_dtype=None, out=None, stream=None):
    """codes (rows x cols/2) + scales (rows x cols/16) + alpha (one-element
    float32 device tensor or view) -> rows x cols float32 / bfloat16."""
    import torch
    rows, half = q.shape
    cols = 2 * half
    if not q.is_cuda:
        raise ValueError(f"q must be a CUDA tensor (got {q.device})")
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or torch.float32, device=q.device)
    _on_device(q.device, s=s, alpha=alpha, out=out)
    bf16 = 1 if out.dtype == torch.bfloat16 else 0
    with torch.cuda.device(q.device):
        _check(lib().nvfp4_dequantize(_ptr(q), _ptr(s), _ptr(alpha), rows, cols, bf16, _ptr(out),
                                      _stream_handle(stream)), "nvfp4_dequantize")
    return out


def nvfp4_error_histogram(x, q_row, s_row, alpha, nbins: int = 24, out=None, stream=None):
    """int64 [3, nbins] device tensor: per bin of v = 6|x|/b (b = block max)
    the element count, the sum of e = 6|x - x^|/b (units 2^-24) and of e*e
    (units 2^-32) for a rowwise copy (plain scale layout); `alpha` is a
    one-element device view of that copy's alpha.  Added to `out` if given."""
    import torch
    p, M, N, ld = _matrix(x)
    if out is None:
        out = torch.zeros((3, nbins), dtype=torch.int64, device=x.device)
    _on_device(x.device, q_row=q_row, s_row=s_row, alpha=alpha, out=out)
    with torch.cuda.device(x.device):
        _check(lib().nvfp4_error_histogram(p, M, N, ld, _ptr(q_row), _ptr(s_row), _ptr(alpha), nbins, _ptr(out),
                                           _stream_handle(stream)), "nvfp4_error_histogram")
    return out


def nvfp4_gemm(qa, sfa, alpha_a, qb, sfb, alpha_b, out=None, out_dtype=None, status=None, stream=None):
    """D (M x N, float32 or bfloat16) = alpha_a * alpha_b * A * B^T: qa (M x K/2) /
    qb (N x K/2) codes with K contiguous, sfa / sfb their scales in the tiled
    layout (NVFP4_SF_SWIZZLED), alpha_a / alpha_b one-element device views of
    the copies' alpha."""
    import torch
    M, half = qa.shape
    N = qb.shape[0]
    K = 2 * half
    if qb.shape[1] != half:
        raise ValueError("A and B must have the same K")
    if not qa.is_cuda:
        raise ValueError(f"qa must be a CUDA tensor (got {qa.device})")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=qa.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _on_device(qa.device, sfa=sfa, alpha_a=alpha_a, qb=qb, sfb=sfb, alpha_b=alpha_b, out=out, status=status)
    bf16 = 1 if out.dtype == torch.bfloat16 else 0
    with torch.cuda.device(qa.device):
        _check(lib().nvfp4_gemm(_ptr(qa), _ptr(sfa), _ptr(alpha_a), _ptr(qb), _ptr(sfb), _ptr(alpha_b), M, N, K,
                                bf16, _ptr(out), out.stride(0), _ptr(status), _stream_handle(stream)), "nvfp4_gemm")
    return out
