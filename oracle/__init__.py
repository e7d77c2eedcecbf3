"""CPU oracle for the NVFP4 training quantizer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and the two share no code.

Two independent CPU implementations live here:

* ``nvfp4_oracle.c`` -- the plain C oracle (built by :func:`build` with
  ``-O2 -ffp-contract=off``), wrapped below with ctypes;
* ``brute.py`` -- a tiny numpy brute-force reference (nearest grid point by
  enumeration, E4M3 by enumeration of all codes, Philox in numpy uint32,
  the Hadamard matrix from scipy) used to pin the C oracle on tiny tensors.

Method sources: "Pretraining Large Language Models with NVFP4" (gist.science
summary of arXiv 2509.25149, section 2) and "Four Over Six (4/6)" (gist.science
technical summary of arXiv 2512.02010, Problem statement, Methodology,
Implementation details).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4_oracle.so")

# interface values (the same integers the library uses; written out again here)
ROWWISE, COLWISE, TWO_D, RHT_ROW, RHT_COL, SR, FOUR_SIX = 1, 2, 4, 8, 16, 32, 64
SEL_MAE, SEL_MSE, SEL_MAXERR = 0, 1, 2
OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_FLAGS, ERR_NONFINITE, ERR_RANGE = 0, -1, -2, -3, -4, -6, -7

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build``.  Plain gcc, no fast-math and
    no FMA contraction, so every float operation rounds exactly as written."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(os.path.join(_HERE, "nvfp4_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        c = ctypes
        L.nvfp4ref_bf16_to_f32.restype = c.c_float
        L.nvfp4ref_bf16_to_f32.argtypes = [c.c_uint16]
        L.nvfp4ref_e2m1_value.restype = c.c_float
        L.nvfp4ref_e2m1_value.argtypes = [c.c_int]
        L.nvfp4ref_round_rn.restype = c.c_int
        L.nvfp4ref_round_rn.argtypes = [c.c_float]
        L.nvfp4ref_round_sr.restype = c.c_int
        L.nvfp4ref_round_sr.argtypes = [c.c_float, c.c_uint32]
        L.nvfp4ref_e4m3_encode.restype = c.c_uint8
        L.nvfp4ref_e4m3_encode.argtypes = [c.c_float]
        L.nvfp4ref_e4m3_value.restype = c.c_float
        L.nvfp4ref_e4m3_value.argtypes = [c.c_uint8]
        L.nvfp4ref_philox4x32_10.restype = None
        L.nvfp4ref_philox4x32_10.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p]
        L.nvfp4ref_rht_signs.restype = c.c_uint16
        L.nvfp4ref_rht_signs.argtypes = [c.c_uint64]
        L.nvfp4ref_hadamard16.restype = c.c_int
        L.nvfp4ref_hadamard16.argtypes = [c.c_int, c.c_int]
        L.nvfp4ref_rht16.restype = None
        L.nvfp4ref_rht16.argtypes = [c.c_void_p, c.c_uint16, c.c_void_p]
        L.nvfp4ref_tree_sum.restype = c.c_float
        L.nvfp4ref_tree_sum.argtypes = [c.c_void_p, c.c_int]
        L.nvfp4ref_quant_block.restype = None
        L.nvfp4ref_quant_block.argtypes = [c.c_void_p, c.c_int, c.c_float, c.c_int, c.c_void_p,
                                           c.c_void_p, c.c_void_p, c.c_void_p]
        L.nvfp4ref_block_error.restype = c.c_float
        L.nvfp4ref_block_error.argtypes = [c.c_void_p, c.c_int, c.c_void_p, c.c_float, c.c_int]
        L.nvfp4ref_amax.restype = c.c_int
        L.nvfp4ref_amax.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_uint32,
                                    c.c_uint64, c.c_void_p]
        L.nvfp4ref_quantize_rows.restype = c.c_int
        L.nvfp4ref_quantize_rows.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p,
                                             c.c_uint32, c.c_int, c.c_uint64, c.c_uint64, c.c_uint64,
                                             c.c_int64, c.c_int64, c.c_void_p, c.c_void_p, c.c_void_p,
                                             c.c_void_p, c.c_void_p]
        L.nvfp4ref_quantize.restype = c.c_int
        L.nvfp4ref_quantize.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p,
                                        c.c_uint32, c.c_int, c.c_uint64, c.c_uint64, c.c_uint64,
                                        c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p]
        L.nvfp4ref_error_histogram.restype = c.c_int
        L.nvfp4ref_error_histogram.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p, c.c_void_p,
                                               c.c_float, c.c_int, c.c_void_p]
        L.nvfp4ref_gemm.restype = c.c_int
        L.nvfp4ref_gemm.argtypes = [c.c_void_p, c.c_void_p, c.c_float, c.c_void_p, c.c_void_p, c.c_float,
                                    c.c_int64, c.c_int64, c.c_int64, c.c_void_p]
        L.nvfp4ref_dequantize.restype = c.c_int
        L.nvfp4ref_dequantize.argtypes = [c.c_void_p, c.c_void_p, c.c_float, c.c_int64, c.c_int64,
                                          c.c_int, c.c_void_p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalar pins
def e2m1_value(idx: int) -> float:
    return lib().nvfp4ref_e2m1_value(idx)


def round_rn(m: float) -> int:
    return lib().nvfp4ref_round_rn(m)


def round_sr(m: float, word: int) -> int:
    return lib().nvfp4ref_round_sr(m, word)


def e4m3_encode(t: float) -> int:
    return lib().nvfp4ref_e4m3_encode(t)


def e4m3_value(e: int) -> float:
    return lib().nvfp4ref_e4m3_value(e)


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().nvfp4ref_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rht_signs(seed: int) -> int:
    return lib().nvfp4ref_rht_signs(seed)


def hadamard16(i: int, j: int) -> int:
    return lib().nvfp4ref_hadamard16(i, j)


def rht16(x, signs: int) -> np.ndarray:
    xx = np.ascontiguousarray(x, dtype=np.float32)
    assert xx.shape == (16,)
    y = np.zeros(16, dtype=np.float32)
    lib().nvfp4ref_rht16(_ptr(xx), signs, _ptr(y))
    return y


def tree_sum(a) -> float:
    aa = np.ascontiguousarray(a, dtype=np.float32)
    return lib().nvfp4ref_tree_sum(_ptr(aa), aa.size)


def quant_block(z, alpha: float, Q: int, words=None):
    """-> (codes uint8[n], scale byte, d)"""
    zz = np.ascontiguousarray(z, dtype=np.float32)
    n = zz.size
    codes = np.zeros(n, dtype=np.uint8)
    e = np.zeros(1, dtype=np.uint8)
    d = np.zeros(1, dtype=np.float32)
    w = None if words is None else np.ascontiguousarray(words, dtype=np.uint32)
    lib().nvfp4ref_quant_block(_ptr(zz), n, alpha, Q, _ptr(w), _ptr(codes), _ptr(e), _ptr(d))
    return codes, int(e[0]), float(d[0])


def block_error(z, codes, d: float, sel: int) -> float:
    zz = np.ascontiguousarray(z, dtype=np.float32)
    cc = np.ascontiguousarray(codes, dtype=np.uint8)
    return lib().nvfp4ref_block_error(_ptr(zz), zz.size, _ptr(cc), d, sel)


# --------------------------------------------------------------- tensor calls
def amax(x_bf16: np.ndarray, flags: int, rht_seed: int = 0, N: int | None = None):
    """x_bf16: uint16 (M, ld) holding an M x N tensor (N defaults to ld).
    Returns (status, float32[2]) -- [rowwise copy, columnwise copy]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, ld = x.shape
    if N is None:
        N = ld
    out = np.zeros(2, dtype=np.float32)
    st = lib().nvfp4ref_amax(_ptr(x), M, N, ld, flags, rht_seed, _ptr(out))
    return st, out


def output_buffers(M: int, N: int, flags: int):
    do_row = bool(flags & ROWWISE)
    do_col = bool(flags & COLWISE)
    q_row = np.zeros((M, N // 2), np.uint8) if do_row else None
    s_row = np.zeros((M, N // 16), np.uint8) if do_row else None
    q_col = np.zeros((N, M // 2), np.uint8) if do_col else None
    s_col = np.zeros((N, M // 16), np.uint8) if do_col else None
    return q_row, s_row, q_col, s_col


def quantize(x_bf16: np.ndarray, N: int, amax2, flags: int, sel: int = SEL_MAE, sr_seed: int = 0,
             rht_seed: int = 0, counter_offset: int = 0, row0: int = 0, row1: int | None = None,
             outs=None):
    """x_bf16: uint16 (M, ld).  Returns dict(status, alpha, q_row, s_row, q_col, s_col)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, ld = x.shape
    if row1 is None:
        row1 = M
    a = np.ascontiguousarray(amax2, dtype=np.float32)
    if outs is None:
        outs = output_buffers(M, N, flags)
    q_row, s_row, q_col, s_col = outs
    alpha = np.zeros(2, dtype=np.float32)
    st = lib().nvfp4ref_quantize_rows(_ptr(x), M, N, ld, _ptr(a), flags, sel, sr_seed, rht_seed,
                                      counter_offset, row0, row1, _ptr(q_row), _ptr(s_row),
                                      _ptr(q_col), _ptr(s_col), _ptr(alpha))
    return dict(status=st, alpha=alpha, q_row=q_row, s_row=s_row, q_col=q_col, s_col=s_col)


def dequantize(q: np.ndarray, s: np.ndarray, alpha: float, rows: int, cols: int,
               out_bf16: bool = False):
    qq = np.ascontiguousarray(q, dtype=np.uint8)
    ss = np.ascontiguousarray(s, dtype=np.uint8)
    out = np.zeros((rows, cols), dtype=np.uint16 if out_bf16 else np.float32)
    st = lib().nvfp4ref_dequantize(_ptr(qq), _ptr(ss), alpha, rows, cols, int(out_bf16), _ptr(out))
    assert st == OK, st
    return out


def error_histogram(x_bf16: np.ndarray, N: int, q_row: np.ndarray, s_row: np.ndarray, alpha: float,
                    nbins: int = 24) -> np.ndarray:
    """uint64 [3, nbins]: counts, sums of e (units 2^-24), sums of e*e (units
    2^-32) per bin of v = 6|x|/b for a rowwise copy (plain scale layout)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, ld = x.shape
    q = np.ascontiguousarray(q_row, dtype=np.uint8)
    s = np.ascontiguousarray(s_row, dtype=np.uint8)
    hist = np.zeros((3, nbins), dtype=np.uint64)
    st = lib().nvfp4ref_error_histogram(_ptr(x), M, N, ld, _ptr(q), _ptr(s), float(alpha), nbins, _ptr(hist))
    assert st == OK, st
    return hist


def gemm(qa: np.ndarray, sa: np.ndarray, alpha_a: float, qb: np.ndarray, sb: np.ndarray, alpha_b: float,
         K: int) -> np.ndarray:
    """D = A * B^T (float32 M x N) of NVFP4 operands with plain scales:
    qa M x K/2 codes, sa M x K/16 scales; qb N x K/2, sb N x K/16."""
    a = np.ascontiguousarray(qa, dtype=np.uint8)
    b = np.ascontiguousarray(qb, dtype=np.uint8)
    xa = np.ascontiguousarray(sa, dtype=np.uint8)
    xb = np.ascontiguousarray(sb, dtype=np.uint8)
    M, N = a.shape[0], b.shape[0]
    d = np.zeros((M, N), dtype=np.float32)
    st = lib().nvfp4ref_gemm(_ptr(a), _ptr(xa), float(alpha_a), _ptr(b), _ptr(xb), float(alpha_b), M, N, K, _ptr(d))
    assert st == OK, st
    return d
