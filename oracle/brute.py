"""Brute-force numpy reference for tiny tensors -- TEST INFRASTRUCTURE ONLY.

A second CPU implementation of the NVFP4 quantizer, written independently of
``nvfp4_oracle.c`` so that the two can pin each other on tiny inputs:

* E2M1 rounding picks the nearest of the eight grid magnitudes by enumerating
  all of them ("Four Over Six (4/6)" technical summary, Problem statement:
  steps 0.5 / 1 / 2 on [0,2] / [2,4] / [4,6]); ties go to the even code.
* E4M3 encoding enumerates every finite non-negative E4M3 value.
* Philox4x32-10 (Salmon et al., SC'11) is vectorised numpy uint32 code.
* The Hadamard matrix is scipy's (Sylvester construction), not a formula.
* 4/6 errors are formed exactly with rationals and rounded once to float32.

Everything is slow and meant for tensors of a few thousand elements.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

ROWWISE, COLWISE, TWO_D, RHT_ROW, RHT_COL, SR, FOUR_SIX = 1, 2, 4, 8, 16, 32, 64
SEL_MAE, SEL_MSE, SEL_MAXERR = 0, 1, 2


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------- E2M1 grid
def e2m1_round_nearest(m: np.ndarray) -> np.ndarray:
    """m >= 0 (float32) -> grid index; nearest by enumeration, ties -> even index."""
    m64 = np.asarray(m, dtype=np.float64)[..., None]
    dist = np.abs(m64 - GRID)                      # (..., 8), exact in float64
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    odd = (np.arange(8) % 2).astype(bool)
    # prefer an even index among the tied candidates
    even_ok = cand & ~odd
    pick_even = even_ok.any(axis=-1)
    idx_even = np.argmax(even_ok, axis=-1)
    idx_any = np.argmax(cand, axis=-1)
    return np.where(pick_even, idx_even, idx_any).astype(np.uint8)


def e2m1_round_stochastic(m: np.ndarray, words: np.ndarray) -> np.ndarray:
    """Grid neighbours lo <= m < hi; round up iff (word>>8)/2^24 < (m-lo)/(hi-lo)."""
    m64 = np.asarray(m, dtype=np.float64)
    lo = np.searchsorted(GRID, m64, side="right") - 1
    lo = np.clip(lo, 0, 7)
    on_grid = (GRID[lo] == m64) | (lo == 7)
    hi = np.minimum(lo + 1, 7)
    span = GRID[hi] - GRID[lo]
    span = np.where(span == 0, 1.0, span)
    p = (m64 - GRID[lo]) / span                      # exact: power-of-two span
    u = (np.asarray(words, dtype=np.uint64) >> np.uint64(8)).astype(np.float64) / 2.0**24
    up = (u < p) & ~on_grid
    return np.where(up, hi, lo).astype(np.uint8)


# ----------------------------------------------------------------- E4M3
def _e4m3_table():
    vals = []
    for code in range(0x7F):  # 0x7F is NaN in E4M3
        ex, man = code >> 3, code & 7
        if ex == 0:
            v = man * 2.0**-9
        else:
            v = (1 + man / 8) * 2.0 ** (ex - 7)
        vals.append(v)
    return np.array(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_table()


def e4m3_encode(t: np.ndarray) -> np.ndarray:
    """t >= 0 -> nearest finite E4M3 code (ties -> even mantissa), saturating at 448."""
    t64 = np.asarray(t, dtype=np.float64)[..., None]
    dist = np.abs(t64 - E4M3_VALUES)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    codes = np.arange(E4M3_VALUES.size)
    even_ok = cand & (codes % 2 == 0)
    pick_even = even_ok.any(axis=-1)
    out = np.where(pick_even, np.argmax(even_ok, axis=-1), np.argmax(cand, axis=-1))
    return out.astype(np.uint8)


# ----------------------------------------------------------------- Philox
_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint32(0x9E3779B9), np.uint32(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr: np.ndarray, key) -> np.ndarray:
    """ctr: uint32 (..., 4); key: (k0, k1).  Returns uint32 (..., 4)."""
    c = np.array(ctr, dtype=np.uint32, copy=True)
    k0 = np.uint32(key[0])
    k1 = np.uint32(key[1])
    with np.errstate(over="ignore"):
        for r in range(10):
            if r:
                k0 = np.uint32(k0 + _W0)
                k1 = np.uint32(k1 + _W1)
            p0 = c[..., 0].astype(np.uint64) * _M0
            p1 = c[..., 2].astype(np.uint64) * _M1
            hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
            lo0 = (p0 & _MASK).astype(np.uint32)
            hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
            lo1 = (p1 & _MASK).astype(np.uint32)
            c = np.stack([hi1 ^ c[..., 1] ^ k0, lo1, hi0 ^ c[..., 3] ^ k1, lo0], axis=-1)
    return c


def element_words(seed: int, offset: int, M: int, N: int) -> np.ndarray:
    """Philox words for every element of an M x N tensor, counter = element index."""
    idx = (np.uint64(offset) + np.arange(M * N, dtype=np.uint64)).reshape(M, N)
    ctr = np.zeros((M, N, 4), dtype=np.uint32)
    ctr[..., 0] = (idx & _MASK).astype(np.uint32)
    ctr[..., 1] = (idx >> np.uint64(32)).astype(np.uint32)
    return philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))


def rht_sign_vector(seed: int) -> np.ndarray:
    w = philox4x32_10(np.array([0, 0, 0, 1], dtype=np.uint32), (seed & 0xFFFFFFFF, seed >> 32))
    bits = (int(w[0]) >> np.arange(16)) & 1
    return np.where(bits == 1, -1.0, 1.0)


def rht(vectors: np.ndarray, seed: int) -> np.ndarray:
    """vectors (..., 16) float32 -> (1/4) H16 diag(s) v, float64 then rounded to float32."""
    from scipy.linalg import hadamard
    H = hadamard(16).astype(np.float64)
    s = rht_sign_vector(seed)
    y = (vectors.astype(np.float64) * s) @ H.T * 0.25
    return y.astype(np.float32)


# ----------------------------------------------------------------- blocks
def _round_f32_exact(q: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (ties -> even)."""
    f = np.float32(float(q))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        dist = abs(Fraction(float(cand)) - q)
        key = (dist, int(np.array(cand, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def quant_block(z: np.ndarray, alpha: np.float32, Q: int, words=None):
    """z: float32 (n,).  Same contract as the C oracle's block routine."""
    z = np.asarray(z, dtype=np.float32)
    b = np.float32(np.max(np.abs(z))) if z.size else np.float32(0)
    t = np.float32(0)
    if b > 0:
        den = np.float32(np.float32(Q) * alpha)
        t = np.float32(b / den)
    e = int(e4m3_encode(np.array([t]))[0])
    d = np.float32(np.float32(E4M3_VALUES[e]) * alpha)
    sign = np.signbit(z).astype(np.uint8)
    if d == 0:
        idx = np.zeros(z.size, dtype=np.uint8)
    else:
        inv = np.float32(np.float32(1) / d)
        v = (z * inv).astype(np.float32)
        m = np.minimum(np.abs(v), np.float32(Q))
        idx = e2m1_round_nearest(m) if words is None else e2m1_round_stochastic(m, words)
    return (sign << 3) | idx, e, d


def block_error(z: np.ndarray, codes: np.ndarray, d: np.float32, sel: int) -> np.float32:
    terms = []
    for zi, ci in zip(z, codes):
        val = Fraction(float(GRID[ci & 7])) * (-1 if ci & 8 else 1)
        err = _round_f32_exact(Fraction(float(zi)) - val * Fraction(float(d)))
        terms.append(np.float32(err * err) if sel == SEL_MSE else np.float32(abs(err)))
    terms = np.array(terms, dtype=np.float32)
    if sel == SEL_MAXERR:
        return np.float32(terms.max())
    while terms.size > 1:  # perfect binary tree, adjacent pairs first
        terms = (terms[0::2] + terms[1::2]).astype(np.float32)
    return np.float32(terms[0])


def quantize_block_46(z, alpha, use46, sel, words):
    c6, e6, d6 = quant_block(z, alpha, 6, words)
    if not use46:
        return c6, e6
    c4, e4, d4 = quant_block(z, alpha, 4, words)
    if block_error(z, c4, d4, sel) < block_error(z, c6, d6, sel):
        return c4, e4
    return c6, e6


# ----------------------------------------------------------------- tensors
def pack(codes: np.ndarray) -> np.ndarray:
    """(R, C) codes -> (R, C/2) bytes, even column in the low nibble."""
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def amax(x_bits: np.ndarray, flags: int, rht_seed: int = 0):
    x = bf16_bits_to_f32(x_bits)
    M, N = x.shape
    plain = np.float32(np.abs(x).max()) if x.size else np.float32(0)
    a = [plain, plain]
    if flags & RHT_ROW:
        a[0] = np.float32(np.abs(rht(x.reshape(M, N // 16, 16), rht_seed)).max())
    if flags & RHT_COL:
        cols = x.T.reshape(N, M // 16, 16)
        a[1] = np.float32(np.abs(rht(cols, rht_seed)).max())
    return np.array(a, dtype=np.float32)


def quantize(x_bits: np.ndarray, amax2, flags: int, sel: int = SEL_MAE, sr_seed: int = 0,
             rht_seed: int = 0, counter_offset: int = 0):
    """Whole-tensor brute force.  Returns dict like the C oracle's wrapper."""
    x = bf16_bits_to_f32(x_bits)
    M, N = x.shape
    use46 = bool(flags & FOUR_SIX)
    denom = np.float32(1536.0 if use46 else 2688.0)
    alpha = np.array([np.float32(amax2[0]) / denom, np.float32(amax2[1]) / denom], dtype=np.float32)
    words = element_words(sr_seed, counter_offset, M, N) if flags & SR else None
    out = {"alpha": alpha}
    if flags & TWO_D:
        codes = np.zeros((M, N), np.uint8)
        scales = np.zeros((M // 16, N // 16), np.uint8)
        for tr in range(M // 16):
            for tc in range(N // 16):
                z = x[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16].reshape(256)
                w = None if words is None else words[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16, 0].reshape(256)
                c, e = quantize_block_46(z, alpha[0], use46, sel, w)
                codes[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16] = c.reshape(16, 16)
                scales[tr, tc] = e
        if flags & ROWWISE:
            out["q_row"] = pack(codes)
            out["s_row"] = np.repeat(scales, 16, axis=0)
        if flags & COLWISE:
            out["q_col"] = pack(codes.T.copy())
            out["s_col"] = np.repeat(scales.T, 16, axis=0)
        return out
    if flags & ROWWISE:
        vec = x.reshape(M, N // 16, 16)
        if flags & RHT_ROW:
            vec = rht(vec, rht_seed)
        codes = np.zeros((M, N), np.uint8)
        scales = np.zeros((M, N // 16), np.uint8)
        for r in range(M):
            for kb in range(N // 16):
                w = None if words is None else words[r, 16 * kb:16 * kb + 16, 0]
                c, e = quantize_block_46(vec[r, kb], alpha[0], use46, sel, w)
                codes[r, 16 * kb:16 * kb + 16] = c
                scales[r, kb] = e
        out["q_row"] = pack(codes)
        out["s_row"] = scales
    if flags & COLWISE:
        vec = x.T.reshape(N, M // 16, 16)
        if flags & RHT_COL:
            vec = rht(vec, rht_seed)
        codes = np.zeros((N, M), np.uint8)
        scales = np.zeros((N, M // 16), np.uint8)
        for c_ in range(N):
            for kb in range(M // 16):
                w = None if words is None else words[16 * kb:16 * kb + 16, c_, 1]
                c, e = quantize_block_46(vec[c_, kb], alpha[1], use46, sel, w)
                codes[c_, 16 * kb:16 * kb + 16] = c
                scales[c_, kb] = e
        out["q_col"] = pack(codes)
        out["s_col"] = scales
    return out
