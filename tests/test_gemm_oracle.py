"""Pins of the oracle's NVFP4 GEMM (D = A * B^T of two operands in the
quantizer's layout, "NVFP4 revolutionizes AI training" headline page: FP4
matrix products on Blackwell).  The oracle dequantizes both operands and sums
the products in double; these tests pin it to facts it does not compute
itself: an exact rational sum built from brute.py's own decoders (grid and
E4M3 tables by enumeration), a closed form, bilinearity in the scales, sign
symmetry and transpose symmetry.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import brute


def _operand(rng, rows, K, scale_lo=0x20, scale_hi=0x48):
    """Random codes (every nibble, both signs) and scale bytes."""
    q = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    s = rng.integers(scale_lo, scale_hi, size=(rows, K // 16), dtype=np.uint8)
    return q, s


def _values_exact(q, s, alpha):
    """Fractions x[r][k] = val(code) * fl32(E4M3(s) * alpha), rounded to float32
    the way a dequantized operand is, from brute.py's tables."""
    rows, half = q.shape
    K = 2 * half
    out = [[None] * K for _ in range(rows)]
    for r in range(rows):
        for k in range(K):
            b = int(q[r, k // 2])
            code = (b & 15) if k % 2 == 0 else (b >> 4)
            val = Fraction(brute.GRID[code & 7]) * (-1 if code & 8 else 1)
            d = brute._round_f32_exact(Fraction(float(brute.E4M3_VALUES[int(s[r, k // 16])])) * Fraction(float(alpha)))
            out[r][k] = Fraction(float(brute._round_f32_exact(val * Fraction(float(d)))))
    return out


def test_gemm_equals_the_exact_rational_sum(ref=oracle):
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 48
    alpha_a, alpha_b = np.float32(0.0371), np.float32(1.9e-3)
    qa, sa = _operand(rng, M, K)
    qb, sb = _operand(rng, N, K)
    d = ref.gemm(qa, sa, alpha_a, qb, sb, alpha_b, K)
    xa, xb = _values_exact(qa, sa, alpha_a), _values_exact(qb, sb, alpha_b)
    for m in range(M):
        for n in range(N):
            exact = sum(xa[m][k] * xb[n][k] for k in range(K))
            want = brute._round_f32_exact(exact)
            assert np.float32(d[m, n]).view(np.uint32) == np.float32(want).view(np.uint32), (m, n, d[m, n], want)


@pytest.mark.parametrize("ea,eb", [(0x38, 0x38), (0x30, 0x41), (0x01, 0x7E)])
def test_gemm_closed_form_for_constant_operands(ea, eb, ref=oracle):
    """Every code is grid value 1.0 (nibble 2): D = K * fl(E4M3(ea)*alpha_a) * fl(E4M3(eb)*alpha_b)."""
    M, N, K = 2, 3, 64
    alpha_a, alpha_b = np.float32(0.5), np.float32(0.125)
    qa = np.full((M, K // 2), 0x22, np.uint8)
    qb = np.full((N, K // 2), 0x22, np.uint8)
    sa = np.full((M, K // 16), ea, np.uint8)
    sb = np.full((N, K // 16), eb, np.uint8)
    d = ref.gemm(qa, sa, alpha_a, qb, sb, alpha_b, K)
    da = np.float32(brute.E4M3_VALUES[ea]) * alpha_a
    db = np.float32(brute.E4M3_VALUES[eb]) * alpha_b
    want = np.float32(K * float(da) * float(db))
    assert np.all(d == want), (d, want)


def test_gemm_is_bilinear_in_scales_and_signs(ref=oracle):
    """Doubling every scale of A (E4M3 code + 8, one exponent step) doubles D
    exactly; flipping the sign bit of every code of B negates D."""
    rng = np.random.default_rng(9)
    M, N, K = 5, 6, 96
    qa, sa = _operand(rng, M, K, 0x20, 0x40)
    qb, sb = _operand(rng, N, K)
    d = ref.gemm(qa, sa, 0.25, qb, sb, 0.75, K)
    d2 = ref.gemm(qa, sa + np.uint8(8), 0.25, qb, sb, 0.75, K)
    assert np.array_equal(d2, 2 * d)
    dn = ref.gemm(qa, sa, 0.25, qb ^ np.uint8(0x88), sb, 0.75, K)
    assert np.array_equal(dn, -d)
    assert np.abs(d).max() > 0


def test_gemm_transpose_symmetry_and_reduction_order(ref=oracle):
    """gemm(B, A) = gemm(A, B)^T bit for bit; against float64 matmul of the
    dequantized operands the result agrees to float32 rounding, and reversing
    the k order of only one operand changes it."""
    rng = np.random.default_rng(11)
    M, N, K = 7, 9, 160
    qa, sa = _operand(rng, M, K)
    qb, sb = _operand(rng, N, K)
    d = ref.gemm(qa, sa, 0.3, qb, sb, 0.02, K)
    assert np.array_equal(ref.gemm(qb, sb, 0.02, qa, sa, 0.3, K), d.T)
    xa = ref.dequantize(qa, sa, 0.3, M, K).astype(np.float64)
    xb = ref.dequantize(qb, sb, 0.02, N, K).astype(np.float64)
    np.testing.assert_allclose(d, (xa @ xb.T).astype(np.float32), rtol=2e-7, atol=1e-30)
    assert not np.allclose(d, (xa @ xb[:, ::-1].T).astype(np.float32), rtol=1e-3)


def test_gemm_rejects_bad_shapes(ref=oracle):
    L = ref.lib()
    assert L.nvfp4ref_gemm(None, None, 1.0, None, None, 1.0, 4, 4, 24, None) == ref.ERR_SHAPE
    assert L.nvfp4ref_gemm(None, None, 1.0, None, None, 1.0, 0, 4, 32, None) == ref.OK
