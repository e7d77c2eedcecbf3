"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here re-types the oracle's formulas: each test checks the oracle
against an outside fact -- a value printed on the pages (tests/golden), a
library routine (ml_dtypes, scipy), a closed form, an invariant, or the
independent brute-force reference in oracle/brute.py.
"""
import numpy as np
import pytest

from conftest import golden_lines
from oracle import brute

ROW, COL, TWO_D, RHT_ROW, RHT_COL, SR, F46 = 1, 2, 4, 8, 16, 32, 64


def bf16_exact(a):
    """round float32 values to bf16 and back (so they are valid inputs)"""
    u = np.asarray(a, dtype=np.float32).view(np.uint32)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return brute.bf16_bits_to_f32(u), u


# ------------------------------------------------------------ E2M1 grid + RN
def test_grid_follows_printed_steps(ref):
    rows = [r for r in golden_lines("e2m1_steps.txt") if r[0] != "range"]
    grid = [0.0]
    for lo, hi, step in rows:
        v = float(lo)
        while v < float(hi):
            v += float(step)
            grid.append(v)
    assert grid == [ref.e2m1_value(i) for i in range(8)]
    rng = [r for r in golden_lines("e2m1_steps.txt") if r[0] == "range"][0]
    assert max(grid) == float(rng[2]) == -float(rng[1])


def test_rn_matches_ml_dtypes(ref):
    ml = pytest.importorskip("ml_dtypes")
    rs = np.random.default_rng(1)
    grid = np.array([ref.e2m1_value(i) for i in range(8)], np.float32)
    mids = (grid[1:] + grid[:-1]) / 2
    sweep = np.concatenate([np.linspace(0, 6, 6001, dtype=np.float32), mids,
                            np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(7)),
                            rs.uniform(0, 6, 4000).astype(np.float32)])
    want = sweep.astype(ml.float4_e2m1fn).view(np.uint8) & 7
    got = np.array([ref.round_rn(float(m)) for m in sweep])
    assert np.array_equal(got, want)
    assert np.array_equal(brute.e2m1_round_nearest(sweep), want)


def test_rn_ties_go_to_even_code(ref):
    # midpoints between grid neighbours; the even code wins
    for m, want in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert ref.round_rn(m) == want, m


# ------------------------------------------------------------ E4M3
def _e4m3_sweep():
    vals = brute.E4M3_VALUES
    mids = (vals[1:] + vals[:-1]) / 2
    rs = np.random.default_rng(2)
    t = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        rs.uniform(0, 448, 20000), np.exp(rs.uniform(np.log(1e-5), np.log(448), 20000)),
                        [0.0, 2.0**-10, 2.0**-11, 1e-30, 2.0**-126]]).astype(np.float32)
    return t[t < 448]


def test_e4m3_encode_matches_ml_dtypes(ref):
    ml = pytest.importorskip("ml_dtypes")
    t = _e4m3_sweep()
    want = t.astype(ml.float8_e4m3fn).view(np.uint8)
    got = np.array([ref.e4m3_encode(float(v)) for v in t], dtype=np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(brute.e4m3_encode(t), want)


def test_e4m3_encode_matches_torch(ref):
    import torch
    t = _e4m3_sweep()
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([ref.e4m3_encode(float(v)) for v in t], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_saturates_at_448(ref):
    facts = dict((r[0], r[1:]) for r in golden_lines("four_over_six_facts.txt"))
    e4m3_max = float(facts["e4m3_max"][0])
    assert ref.e4m3_value(0x7E) == e4m3_max
    for t in [448.0, 463.9, 464.0, 470.0, 480.0, 672.0, 1e6, 3e38]:
        assert ref.e4m3_encode(t) == 0x7E
    assert ref.e4m3_encode(447.0) == 0x7E and ref.e4m3_encode(410.0) == 0x7D
    assert ref.e4m3_encode(400.0) == 0x7C                # tie between 384 and 416: even mantissa


def test_e4m3_decode_all_codes(ref):
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(0x7F, dtype=np.uint8)
    want = codes.view(ml.float8_e4m3fn).astype(np.float32)
    got = np.array([ref.e4m3_value(int(c)) for c in codes], np.float32)
    assert np.array_equal(got, want)


# ------------------------------------------------------------ worked facts of the 4/6 page
def test_four_is_two_thirds_of_block_max_at_scale_six(ref):
    facts = dict((r[0], r[1:]) for r in golden_lines("four_over_six_facts.txt"))
    frac = float(facts["four_at_scale_six_fraction"][0])
    alpha = np.float32(0.125)               # power of two: every scale below is exact
    b = np.float32(0.75)                    # t = b / (6 alpha) = 1 -> e = 1.0, d = alpha
    z = np.zeros(16, np.float32)
    z[0] = b
    z[1] = np.float32(4) * alpha            # the FP4 value "4" at this block scale
    codes, e, d = ref.quant_block(z, float(alpha), 6)
    assert d == alpha and codes[0] == 7 and codes[1] == 6
    assert abs(z[1] / b - frac) < 1e-3
    # no representable magnitude lies strictly between 66.6% and 100% of the max
    mags = sorted({ref.e2m1_value(i) * d / b for i in range(8)})
    assert [m for m in mags if 2 / 3 + 1e-9 < m < 1 - 1e-9] == []
    for fraction in np.linspace(0.67, 0.99, 33):
        zz = z.copy()
        zz[1] = np.float32(fraction) * b
        c, _, _ = ref.quant_block(zz, float(alpha), 6)
        assert ref.e2m1_value(c[1] & 7) in (4.0, 6.0)


def test_value_at_75_percent_is_exact_three_at_scale_four(ref):
    facts = dict((r[0], r[1:]) for r in golden_lines("four_over_six_facts.txt"))
    frac, q = float(facts["value_fraction_exact_at_scale4"][0]), float(facts["value_fraction_exact_at_scale4"][1])
    alpha = 0.125
    b = np.float32(0.75)
    z = np.full(16, np.float32(frac) * b, np.float32)
    z[0] = b
    c4, e4, d4 = ref.quant_block(z, alpha, 4)
    assert ref.e2m1_value(c4[1] & 7) == q
    assert ref.block_error(z, c4, d4, 0) == 0.0
    # at scale 6 the same value falls into the 4..6 gap: 4.5 rounds to 4, error = max/12
    c6, e6, d6 = ref.quant_block(z, alpha, 6)
    assert ref.e2m1_value(c6[1] & 7) == 4.0
    assert ref.block_error(z[1:2], c6[1:2], d6, 0) == pytest.approx(float(b) / 12, rel=1e-6)


def test_gap_sizes(ref):
    facts = [r for r in golden_lines("four_over_six_facts.txt") if r[0].startswith("gap_")]
    grid = [ref.e2m1_value(i) for i in range(8)]
    for name, a, b_, gap in facts:
        a, b_, gap = float(a), float(b_), float(gap)
        assert a in grid and b_ in grid and b_ - a == gap
        assert not [g for g in grid if a < g < b_]


def test_tensor_scale_headroom_256_vs_448(ref):
    facts = dict((r[0], r[1:]) for r in golden_lines("four_over_six_facts.txt"))
    ratio = float(facts["scale_ratio_4_over_6"][0])
    m46 = float(facts["tensor_scale_max_46"][0])
    A = np.float32(3.0)
    z = np.zeros(16, np.float32)
    z[0] = A                                 # the block that holds the tensor maximum
    a46 = np.float32(A / np.float32(6 * m46))
    _, e6, d6 = ref.quant_block(z, float(a46), 6)
    _, e4, d4 = ref.quant_block(z, float(a46), 4)
    assert ref.e4m3_value(e6) == 256.0 and ref.e4m3_value(e4) == 384.0
    assert ref.e4m3_value(e4) / ref.e4m3_value(e6) == ratio      # no overflow with 256
    a448 = np.float32(A / np.float32(2688))
    _, e6, _ = ref.quant_block(z, float(a448), 6)
    _, e4, _ = ref.quant_block(z, float(a448), 4)
    assert ref.e4m3_value(e6) == 448.0
    assert ref.e4m3_value(e4) == 448.0 and 1.5 * 448.0 > 448.0   # 672 saturates with 448


def test_46_keeps_four_for_the_75_percent_block_and_six_for_an_exact_block(ref):
    alpha = 0.125
    b = np.float32(0.75)
    z75 = np.full(16, np.float32(0.75) * b, np.float32)
    z75[0] = b
    zexact = np.full(16, np.float32(alpha), np.float32)   # value 1 at scale 6: exact
    zexact[0] = b
    for sel in (0, 1, 2):
        c6, e6, d6 = ref.quant_block(z75, alpha, 6)
        c4, e4, d4 = ref.quant_block(z75, alpha, 4)
        assert ref.block_error(z75, c4, d4, sel) < ref.block_error(z75, c6, d6, sel)
        c6, e6, d6 = ref.quant_block(zexact, alpha, 6)
        c4, e4, d4 = ref.quant_block(zexact, alpha, 4)
        assert ref.block_error(zexact, c6, d6, sel) == 0.0
        assert ref.block_error(zexact, c4, d4, sel) > 0.0
    # and through the whole-tensor call: the scale byte records the choice
    x = np.stack([z75] * 8 + [zexact] * 8).astype(np.float32)
    _, bits = bf16_exact(x)
    st, am = ref.amax(bits, ROW | F46)
    out = ref.quantize(bits, 16, am, ROW | F46, sel=0)
    assert out["status"] == 0
    alpha46 = out["alpha"][0]
    _, e_six, _ = ref.quant_block(x[0], float(alpha46), 6)
    _, e_four, _ = ref.quant_block(x[0], float(alpha46), 4)
    assert out["s_row"][0, 0] == e_four and e_four != e_six
    _, e_six, _ = ref.quant_block(x[8], float(alpha46), 6)
    assert out["s_row"][8, 0] == e_six


def test_selection_rules_can_disagree(ref):
    """The three rules named on the page are different rules: random blocks where
    MAE, MSE and MAXERR pick differently exist, and the brute reference agrees."""
    rs = np.random.default_rng(7)
    seen = set()
    for _ in range(3000):
        z, _ = bf16_exact(rs.standard_normal(16) * rs.uniform(0.2, 2))
        picks = []
        for sel in (0, 1, 2):
            c6, e6, d6 = ref.quant_block(z, 0.01, 6)
            c4, e4, d4 = ref.quant_block(z, 0.01, 4)
            s6, s4 = ref.block_error(z, c6, d6, sel), ref.block_error(z, c4, d4, sel)
            assert s6 == brute.block_error(z, c6, np.float32(d6), sel)
            assert s4 == brute.block_error(z, c4, np.float32(d4), sel)
            picks.append(4 if s4 < s6 else 6)
        seen.add(tuple(picks))
        if len(seen) >= 4:
            break
    assert len(seen) >= 3, seen


def test_error_is_original_minus_dequantized(ref):
    """err_i = z_i - dequant(q_i): scores of a block match the dequantizer's output."""
    rs = np.random.default_rng(8)
    z, bits = bf16_exact(rs.standard_normal(16))
    am = np.abs(z).max()
    alpha = np.float32(am / np.float32(2688))
    codes, e, d = ref.quant_block(z, float(alpha), 6)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    xh = ref.dequantize(packed, np.array([[e]], np.uint8), float(alpha), 1, 16)[0]
    # dequant rounds val*d once; the error uses the exact product -- equal here
    # because val*d is exact for these small codes and scales
    exact = np.array([np.float64(zz) - np.float64(x) for zz, x in zip(z, xh)])
    assert ref.block_error(z, codes, d, 2) == pytest.approx(np.abs(exact).max(), rel=1e-6, abs=1e-30)


# ------------------------------------------------------------ tree order
def test_tree_sum_is_adjacent_pairs_first(ref):
    assert ref.tree_sum([1e8, 1, -1e8, 1]) == 0.0            # ((1e8+1) + (-1e8+1)) in fp32
    assert ref.tree_sum([1e8, -1e8, 1, 1]) == 2.0
    rs = np.random.default_rng(9)
    for n in (16, 256):
        a = (rs.standard_normal(n) * 10 ** rs.uniform(-3, 3, n)).astype(np.float32)
        t = a.copy()
        while t.size > 1:
            t = (t[0::2] + t[1::2]).astype(np.float32)
        assert ref.tree_sum(a) == t[0]


# ------------------------------------------------------------ Hadamard
def test_hadamard_is_sylvester_and_orthogonal(ref):
    from scipy.linalg import hadamard
    H = np.array([[ref.hadamard16(i, j) for j in range(16)] for i in range(16)])
    assert np.array_equal(H, hadamard(16))
    assert np.array_equal(H @ H.T, 16 * np.eye(16, dtype=int))


def test_rht_preserves_norm_inner_products_and_inverts(ref):
    from scipy.linalg import hadamard
    rs = np.random.default_rng(10)
    s = ref.rht_signs(0x5EED)
    sv = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    for _ in range(50):
        x, _ = bf16_exact(rs.standard_t(3, 16))
        w, _ = bf16_exact(rs.standard_normal(16))
        y = ref.rht16(x, s).astype(np.float64)
        v = ref.rht16(w, s).astype(np.float64)
        nx = np.linalg.norm(x.astype(np.float64))
        assert abs(np.linalg.norm(y) - nx) <= 1e-6 * nx
        assert abs(y @ v - x.astype(np.float64) @ w) <= 1e-6 * nx * np.linalg.norm(w)
        back = sv * (hadamard(16) @ y) / 4.0
        assert np.allclose(back, x, rtol=0, atol=1e-6 * nx)
    # all-plus signs reduce to the plain orthonormal Walsh-Hadamard transform
    x, _ = bf16_exact(rs.standard_normal(16))
    plain = (hadamard(16) @ x.astype(np.float64) / 4).astype(np.float32)
    assert np.array_equal(ref.rht16(x, 0), plain)
    # a single spike spreads evenly: |y_i| = |x_0| / 4 for every i
    spike = np.zeros(16, np.float32)
    spike[3] = 8.0
    assert np.array_equal(np.abs(ref.rht16(spike, s)), np.full(16, 2.0, np.float32))


def test_rht_signs_come_from_philox(ref):
    for seed in (0, 1, 0x5EED, 0xDEADBEEFCAFE):
        w = brute.philox4x32_10(np.array([0, 0, 0, 1], np.uint32), (seed & 0xFFFFFFFF, seed >> 32))
        assert ref.rht_signs(seed) == int(w[0]) & 0xFFFF


# ------------------------------------------------------------ Philox
def test_philox_known_answers(ref):
    for row in golden_lines("philox4x32_10_kat.txt"):
        v = [int(h, 16) for h in row]
        assert list(ref.philox4x32_10(v[0:4], v[4:6])) == v[6:10]
        assert list(brute.philox4x32_10(np.array(v[0:4], np.uint32), v[4:6])) == v[6:10]


def test_philox_c_and_numpy_agree(ref):
    rs = np.random.default_rng(11)
    ctr = rs.integers(0, 2**32, (200, 4), dtype=np.uint64).astype(np.uint32)
    for i in range(200):
        key = [int(k) for k in rs.integers(0, 2**32, 2)]
        assert np.array_equal(ref.philox4x32_10(ctr[i], key), brute.philox4x32_10(ctr[i], key))


def test_philox_words_look_uniform(ref):
    w = brute.element_words(0x1234ABCD, 0, 256, 256)[..., 0].ravel()
    counts = np.bincount((w >> 24).astype(np.int64), minlength=256)
    exp = w.size / 256
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)


# ------------------------------------------------------------ stochastic rounding
def test_sr_follows_the_printed_example(ref):
    """1.4 between 1 and 2 rounds up with probability 0.4.  On the E2M1 grid the
    same situation (neighbours one unit apart, 40% of the way) is 2.4 in [2, 3]."""
    value, lower, upper, p_down, p_up = (float(v) for v in golden_lines("stochastic_rounding_example.txt")[0])
    m = 2.0 + (value - lower) / (upper - lower)
    words = brute.element_words(99, 0, 200, 200)[..., 0].ravel()
    up = np.array([ref.round_sr(m, int(w)) for w in words]) == 5
    n = words.size
    assert abs(up.mean() - p_up) < 5 * np.sqrt(p_up * p_down / n)


@pytest.mark.parametrize("m", [0.1, 0.3, 1.2, 1.9, 2.4, 3.7, 4.5, 5.9])
def test_sr_is_unbiased(ref, m):
    m = float(np.float32(m))
    words = brute.element_words(1234, 0, 100, 100)[..., 0].ravel()
    vals = np.array([ref.e2m1_value(ref.round_sr(m, int(w))) for w in words])
    lo = max(g for g in [ref.e2m1_value(i) for i in range(8)] if g <= m)
    hi = min(g for g in [ref.e2m1_value(i) for i in range(8)] if g > m)
    p = (m - lo) / (hi - lo)
    sd = (hi - lo) * np.sqrt(p * (1 - p) / vals.size)
    assert abs(vals.mean() - m) < 5 * sd
    assert set(np.unique(vals)) <= {lo, hi}
    assert np.array_equal([brute.e2m1_round_stochastic(np.float32(m), words)][0],
                          [ref.round_sr(m, int(w)) for w in words])


def test_sr_edge_cases(ref):
    for i in range(8):
        g = ref.e2m1_value(i)
        for w in (0, 0x80000000, 0xFFFFFFFF):
            assert ref.round_sr(g, w) == i            # on the grid: never moves
    assert ref.round_sr(1e-30, 0) == 1                 # u = 0 < p: rounds up
    assert ref.round_sr(0.49, 0xFFFFFFFF) == 0         # u = 1 - 2^-24 >= p: stays
    just_below = float(np.nextafter(np.float32(0.5), 0))    # p = 1 - 2^-24
    assert ref.round_sr(just_below, 0xFFFFFFFF) == 0         # u = p: not below, stays
    assert ref.round_sr(just_below, 0xFFFFFE00) == 1         # u = 1 - 2^-23 < p: up


# ------------------------------------------------------------ whole tensors, brute force
def _tiny_inputs():
    rs = np.random.default_rng(12)
    M, N = 32, 48
    a = rs.standard_normal((M, N)).astype(np.float32)
    a[rs.random((M, N)) < 0.02] *= 40                   # outliers
    a[0:16, 0:16] = 0.0                                 # an all-zero 2D tile / blocks
    a[16, 16:32] *= 1e-7                                # a block far below the tensor max
    a[20, 0] = -0.0
    yield "normal", bf16_exact(a)[1]
    g = (rs.standard_t(3, (48, 32)) * 1e-3).astype(np.float32)
    yield "student_t", bf16_exact(g)[1]


VALID_FLAGS = [f for f in range(128)
               if (f & 3) and not ((f & TWO_D) and (f & (RHT_ROW | RHT_COL)))
               and not ((f & RHT_ROW) and not (f & ROW)) and not ((f & RHT_COL) and not (f & COL))]


@pytest.mark.parametrize("flags", VALID_FLAGS)
def test_oracle_matches_brute_force_on_tiny_tensors(ref, flags):
    sels = (0, 1, 2) if flags & F46 else (0,)
    for name, bits in _tiny_inputs():
        M, N = bits.shape
        st, am = ref.amax(bits, flags, rht_seed=0x5EED)
        assert st == 0
        assert np.array_equal(am, brute.amax(bits, flags, rht_seed=0x5EED))
        for sel in sels:
            got = ref.quantize(bits, N, am, flags, sel=sel, sr_seed=0x1234ABCD, rht_seed=0x5EED,
                               counter_offset=77)
            want = brute.quantize(bits, am, flags, sel=sel, sr_seed=0x1234ABCD, rht_seed=0x5EED,
                                  counter_offset=77)
            assert got["status"] == 0
            assert np.array_equal(got["alpha"], want["alpha"])
            for k in ("q_row", "s_row", "q_col", "s_col"):
                if k in want:
                    assert np.array_equal(got[k], want[k]), (name, flags, sel, k)


def test_2d_copies_are_transposes_and_dequantize_identically(ref):
    bits = synthetic_weight(64, 96)
    st, am = ref.amax(bits, ROW | COL | TWO_D)
    out = ref.quantize(bits, 96, am, ROW | COL | TWO_D)
    unpack = lambda q: np.stack([q & 15, q >> 4], -1).reshape(q.shape[0], -1)
    assert np.array_equal(unpack(out["q_col"]), unpack(out["q_row"]).T)
    dr = ref.dequantize(out["q_row"], out["s_row"], out["alpha"][0], 64, 96)
    dc = ref.dequantize(out["q_col"], out["s_col"], out["alpha"][1], 96, 64)
    assert np.array_equal(dc.T.view(np.uint32), dr.view(np.uint32))


def synthetic_weight(M, N):
    import synthetic
    return synthetic.weight(M, N, 5)


def test_dequantize_decodes_grid_times_scale(ref):
    rs = np.random.default_rng(13)
    q = rs.integers(0, 256, (4, 16), dtype=np.uint8)
    s = rs.integers(0, 0x7F, (4, 2), dtype=np.uint8)
    alpha = np.float32(0.37)
    out = ref.dequantize(q, s, float(alpha), 4, 32)
    codes = np.stack([q & 15, q >> 4], -1).reshape(4, 32)
    d = (brute.E4M3_VALUES[np.repeat(s, 16, axis=1)].astype(np.float32) * alpha).astype(np.float32)
    val = (brute.GRID[codes & 7] * np.where(codes & 8, -1, 1)).astype(np.float32)
    assert np.array_equal(out, (val * d).astype(np.float32))
    ob = ref.dequantize(q, s, float(alpha), 4, 32, out_bf16=True)
    import torch
    assert np.array_equal(ob, torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------------ degenerate cases and status
def test_zero_tensor(ref):
    bits = np.zeros((32, 32), np.uint16)
    bits[3, 5] = 0x8000                                  # -0.0
    st, am = ref.amax(bits, ROW | COL)
    assert st == 0 and am[0] == 0 and am[1] == 0
    out = ref.quantize(bits, 32, am, ROW | COL | F46)
    assert out["status"] == 0 and out["alpha"][0] == 0
    assert not out["s_row"].any() and not out["s_col"].any()
    # element (3, 5): odd column -> high nibble of byte 2 of row 3; in the
    # transposed copy odd row -> high nibble of byte 1 of row 5
    assert out["q_row"][3, 2] == 0x80 and out["q_col"][5, 1] == 0x80
    assert out["q_row"].sum() == 0x80 and out["q_col"].sum() == 0x80


def test_empty_tensor(ref):
    bits = np.zeros((0, 32), np.uint16)
    st, am = ref.amax(bits, ROW)
    assert st == 0 and am[0] == 0
    assert ref.quantize(bits, 32, am, ROW)["status"] == 0


def test_status_codes(ref):
    bits = np.zeros((16, 32), np.uint16)
    bits[1, 1] = 0x7F80                                  # +inf
    st, am = ref.amax(bits, ROW)
    assert st == 0 and np.isinf(am[0])
    assert ref.quantize(bits, 32, am, ROW)["status"] == -6
    bits[1, 1] = 0x7FC0                                  # NaN
    st, am = ref.amax(bits, ROW | COL)
    assert np.isnan(am[0]) and ref.quantize(bits, 32, am, ROW | COL)["status"] == -6
    tiny = np.full((16, 32), 0x0001, np.uint16)          # 2^-133: far below 2^-100
    st, am = ref.amax(tiny, ROW)
    assert ref.quantize(tiny, 32, am, ROW)["status"] == -7
    ok = np.zeros((16, 32), np.uint16)
    assert ref.amax(ok, 0)[0] == -4                      # no copy requested
    assert ref.amax(ok, ROW | TWO_D | RHT_ROW)[0] == -4  # 2D with a Hadamard transform
    assert ref.amax(ok, COL | RHT_ROW)[0] == -4          # transform of a copy not requested
    assert ref.amax(np.zeros((8, 32), np.uint16), COL)[0] == -2    # M not a multiple of 16
    assert ref.amax(np.zeros((16, 24), np.uint16), ROW)[0] == -2   # N not a multiple of 16
    assert ref.amax(np.zeros((8, 32), np.uint16), ROW)[0] == 0     # rowwise only: any M


def test_row_stripes_and_counter_offset_reproduce_the_whole(ref):
    import synthetic
    bits = synthetic.gradient(64, 48, 3)
    flags = ROW | COL | SR | RHT_COL
    st, am = ref.amax(bits, flags, rht_seed=9)
    full = ref.quantize(bits, 48, am, flags, sr_seed=5, rht_seed=9)
    outs = ref.output_buffers(64, 48, flags)
    for r0 in range(0, 64, 16):
        ref.quantize(bits, 48, am, flags, sr_seed=5, rht_seed=9, row0=r0, row1=r0 + 16, outs=outs)
    for k, arr in zip(("q_row", "s_row", "q_col", "s_col"), outs):
        assert np.array_equal(arr, full[k])
    # a shard that owns rows 32..63 reproduces them with counter_offset = 32*N
    shard = ref.quantize(bits[32:], 48, am, ROW | SR, sr_seed=5, counter_offset=32 * 48)
    whole = ref.quantize(bits, 48, am, ROW | SR, sr_seed=5)
    assert np.array_equal(shard["q_row"], whole["q_row"][32:])
