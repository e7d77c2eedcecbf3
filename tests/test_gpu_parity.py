"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small cases span several CTA tiles (64 x 256) plus ragged tails.  The recipe's
full-size workloads run in the launch configuration the benchmark times and
are compared element by element with the oracle run on every host core (row
stripes in spawned processes).  Every output buffer is guarded by canary
bytes (gpu_helpers), so stray stores fail too.
"""

import numpy as np
import pytest
import torch

import nvfp4_bit_block_gb300 as nv
import oracle
import synthetic
from gpu_helpers import (assert_copy_exact, assert_parity, gpu_quantize, ref_quantize, selftest_lib, to_device,
                         signed_grid_index)

pytestmark = pytest.mark.gpu

ROW, COL, TWO_D, RHT_ROW, RHT_COL, SR, F46 = 1, 2, 4, 8, 16, 32, 64
VALID_FLAGS = [f for f in range(128)
               if (f & 3) and not ((f & TWO_D) and (f & (RHT_ROW | RHT_COL)))
               and not ((f & RHT_ROW) and not (f & ROW)) and not ((f & RHT_COL) and not (f & COL))]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nv.build()
    oracle.build()


def small_input(M=272, N=528, kind="act"):
    if kind == "act":
        bits = synthetic.activation_outlier_channels(M, N, 11, frac=0.01)
    elif kind == "grad":
        bits = synthetic.gradient(M, N, 12)
    else:
        bits = synthetic.weight(M, N, 13)
    f = bits.view(np.uint16).copy()
    # degenerate blocks: an all-zero 16x16 tile, a tiny block, negative zeros
    f[16:32, 32:48] = 0
    f[40, 64:80] = 0x0001                       # bf16 2^-133 next to O(1) values
    f[50, 100] = 0x8000
    return f


@pytest.mark.parametrize("flags", VALID_FLAGS)
def test_every_flag_combination_small(flags):
    sels = (0, 1, 2) if flags & F46 else (0,)
    kind = "grad" if flags & (SR | RHT_ROW | RHT_COL) else ("weight" if flags & TWO_D else "act")
    bits = small_input(kind=kind)
    x = to_device(bits)
    for sel in sels:
        g = gpu_quantize(x, flags, sel, sr_seed=0x1234ABCD, rht_seed=0x5EED, counter_offset=3)
        r = ref_quantize(bits, flags, sel, sr_seed=0x1234ABCD, rht_seed=0x5EED, counter_offset=3)
        assert_parity(g, r, flags)


@pytest.mark.parametrize("flags", [ROW, ROW | F46, ROW | SR, ROW | RHT_ROW | SR | F46])
@pytest.mark.parametrize("M", [1, 7, 261])
def test_rowwise_only_ragged_rows(flags, M):
    bits = synthetic.activation_outlier_entries(M, 272, 21)
    g = gpu_quantize(to_device(bits), flags, 1, sr_seed=5, rht_seed=6)
    r = ref_quantize(bits, flags, 1, sr_seed=5, rht_seed=6)
    assert_parity(g, r, flags)


@pytest.mark.parametrize("flags", [ROW | COL | F46, ROW | COL | TWO_D, ROW | COL | RHT_COL | SR])
def test_padded_leading_dimension(flags):
    bits = small_input(144, 272)
    x = to_device(bits, ld=312)
    assert x.stride(0) == 312
    g = gpu_quantize(x, flags, 0, sr_seed=1, rht_seed=2)
    r = ref_quantize(bits, flags, 0, sr_seed=1, rht_seed=2)
    assert_parity(g, r, flags)


@pytest.mark.parametrize("shape", [(16, 16), (16, 256), (32, 16), (128, 256), (144, 2064)])
def test_tile_edges(shape):
    bits = synthetic.activation_outlier_channels(*shape, 31, frac=0.05)
    for flags in (ROW | COL | F46, ROW | COL | TWO_D | F46, ROW | COL | RHT_COL | SR):
        g = gpu_quantize(to_device(bits), flags, 2, sr_seed=9, rht_seed=10)
        r = ref_quantize(bits, flags, 2, sr_seed=9, rht_seed=10)
        assert_parity(g, r, flags)


def test_extreme_magnitudes():
    """bf16 values near the top of the range, subnormal inputs and blocks whose
    scale underflows E4M3 (subnormal and zero scale bytes)."""
    rs = np.random.default_rng(3)
    f = (rs.standard_normal((64, 256)) * 1e-3).astype(np.float32)
    f[0, 0] = 3.0e38                                       # amax near bf16 max
    f[1, :16] = 1e30
    f[2, :] = rs.standard_normal(256).astype(np.float32) * 1e-36   # bf16 subnormal range
    bits = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for flags in (ROW | COL, ROW | COL | F46, ROW | COL | TWO_D, ROW | COL | SR, ROW | COL | F46 | SR):
        for sel in (0, 1, 2):
            g = gpu_quantize(to_device(bits), flags, sel, sr_seed=4)
            r = ref_quantize(bits, flags, sel, sr_seed=4)
            assert_parity(g, r, flags)


def test_zero_and_empty_tensors():
    bits = np.zeros((32, 48), np.uint16)
    bits[3, 5] = 0x8000
    for flags in (ROW | COL, ROW | COL | F46 | SR, ROW | COL | TWO_D):
        g = gpu_quantize(to_device(bits), flags)
        r = ref_quantize(bits, flags)
        assert_parity(g, r, flags)
        assert g["alpha"][0] == 0 and not g["s_row"].any()
    empty = torch.zeros((0, 32), dtype=torch.bfloat16, device="cuda")
    amax = nv.nvfp4_amax(empty, ROW)
    out = nv.nvfp4_quantize(empty, amax, ROW)
    torch.cuda.synchronize()
    assert amax.cpu().tolist() == [0.0, 0.0] and out.alpha.cpu().tolist() == [0.0, 0.0]


def test_nonfinite_and_tiny_amax_report_a_status_and_write_nothing():
    """An Inf or NaN anywhere makes the amax (plain, or of the Hadamard-
    transformed copy) non-finite; the quantize then reports NONFINITE and
    writes nothing (every kernel: the 1D round-to-nearest and 4/6 kernels,
    the stochastic-rounding kernel of both copies, 2D)."""
    for flags in (ROW | COL, ROW | COL | RHT_COL, ROW | COL | RHT_ROW | RHT_COL, ROW | COL | SR,
                  ROW | COL | RHT_COL | SR, ROW | COL | F46, ROW | COL | TWO_D):
        for pattern, want in ((0x7F80, -6), (0xFFC0, -6)):
            bits = synthetic.weight(32, 32, 1)
            bits[5, 7] = pattern
            x = to_device(bits)
            amax = nv.nvfp4_amax(x, flags)
            out = nv.Quantized(*(torch.full(s, 0xAB, dtype=torch.uint8, device="cuda")
                                 for s in nv.output_shapes(32, 32, flags)),
                               alpha=torch.zeros(2, device="cuda"), status=torch.zeros(1, dtype=torch.int32,
                                                                                       device="cuda"))
            nv.nvfp4_quantize(x, amax, flags, out=out)
            torch.cuda.synchronize()
            assert out.status.item() == want
            assert not np.isfinite(amax.cpu().numpy()).any()
            assert all(bool((t == 0xAB).all()) for t in (out.q_row, out.s_row, out.q_col, out.s_col))
            st, am = oracle.amax(bits, flags)
            assert not np.isfinite(am).any()
            assert oracle.quantize(bits, 32, am, flags)["status"] == want
    tiny = np.full((32, 32), 0x0001, np.uint16)
    g = gpu_quantize(to_device(tiny), ROW)
    assert g["status"] == -7
    st, am = oracle.amax(tiny, ROW)
    assert oracle.quantize(tiny, 32, am, ROW)["status"] == -7


def relayout_tiled(plain: np.ndarray) -> np.ndarray:
    """Plain R x C scales -> the tiled layout of block-scaled MMA operands,
    from its definition: 128-row x 4-column tiles of 512 bytes in row-major
    tile order over the padded matrix, scale (r, c) at byte
    (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4 of its tile; padding zero."""
    R, C = plain.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * (Cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    out = np.zeros(Rp * Cp, np.uint8)
    out[off] = plain
    return out.reshape(Rp, Cp)


@pytest.mark.parametrize("flags,sel", [(ROW, 0), (ROW | F46, 0), (ROW | F46, 1), (ROW | SR, 0)])
def test_error_histogram_matches_oracle(flags, sel):
    """nvfp4_error_histogram (integer bins) equals the oracle's histogram of the
    same quantized copy, on the small input and on the activation workload."""
    for bits in (small_input(), synthetic.workload("act_46mae_8192x5120") if flags == ROW | F46 else None):
        if bits is None:
            continue
        x = to_device(bits)
        g = gpu_quantize(x, flags, sel, sr_seed=4)
        out = g["_out"]
        h = nv.nvfp4_error_histogram(x, out.q_row, out.s_row, out.alpha[:1], 24).cpu().numpy().astype(np.uint64)
        r = oracle.error_histogram(bits, bits.shape[1], g["q_row"], g["s_row"], float(g["alpha"][0]), 24)
        assert np.array_equal(h, r)
        assert int(h[0].sum()) > 0


def test_relayout_reference_is_a_bijection():
    """The test's relayout places every scale of a padded matrix exactly once."""
    plain = np.arange(256 * 8, dtype=np.int64).reshape(256, 8) % 251 + 1
    tiled = relayout_tiled(plain.astype(np.uint8))
    assert tiled.size == plain.size and np.count_nonzero(tiled) == plain.size
    assert tiled.reshape(-1)[:16].tolist() == [plain[0, 0], plain[0, 1], plain[0, 2], plain[0, 3],
                                               plain[32, 0], plain[32, 1], plain[32, 2], plain[32, 3],
                                               plain[64, 0], plain[64, 1], plain[64, 2], plain[64, 3],
                                               plain[96, 0], plain[96, 1], plain[96, 2], plain[96, 3]]


@pytest.mark.parametrize("flags", [ROW | COL, ROW | COL | F46, ROW | COL | TWO_D, ROW | COL | RHT_COL | SR, ROW, COL])
def test_swizzled_scales_are_the_plain_scales_relaid(flags):
    """NVFP4_SF_SWIZZLED writes each copy's scales in the tiled MMA operand
    layout (padding rows to 128 and scale columns to 4, padding untouched);
    codes are unchanged.  Shapes include partial tiles in both directions."""
    for M, N in ((272, 528), (400, 1040)):
        bits = small_input(M, N)
        x = to_device(bits)
        g = gpu_quantize(x, flags, 1, sr_seed=5, rht_seed=6)
        gs = gpu_quantize(x, flags | nv.SF_SWIZZLED, 1, sr_seed=5, rht_seed=6)
        for which in ("row", "col"):
            if g[f"q_{which}"] is None:
                continue
            assert np.array_equal(gs[f"q_{which}"], g[f"q_{which}"])
            assert np.array_equal(gs[f"s_{which}"], relayout_tiled(g[f"s_{which}"]))


@pytest.mark.parametrize("flags,sel", [(ROW | COL, 0), (ROW | COL | F46, 1), (ROW | COL | RHT_COL | SR, 0),
                                       (ROW | F46 | SR, 2), (COL, 0)])
def test_more_tiles_than_one_round(flags, sel):
    """A 1984 x 4096 tensor has 496 tiles of 64 x 256 (992 of 64 x 128 for
    plain round-to-nearest): more than one round of the persistent grid on
    152 SMs at two, three or four CTAs per SM, and not a multiple of any, so
    CTAs walk different numbers of tiles.  Every code and scale byte equals
    the oracle's, and the tiled scale layout is the plain one relaid."""
    M, N = 1984, 4096
    assert torch.cuda.get_device_properties(0).multi_processor_count * 3 < (M // 64) * (N // 256)
    bits = small_input(M, N, kind="grad" if flags & SR else "act")
    x = to_device(bits)
    g = gpu_quantize(x, flags, sel, sr_seed=21, rht_seed=22, counter_offset=5)
    r = ref_quantize(bits, flags, sel, sr_seed=21, rht_seed=22, counter_offset=5)
    assert_parity(g, r, flags)
    gs = gpu_quantize(x, flags | nv.SF_SWIZZLED, sel, sr_seed=21, rht_seed=22, counter_offset=5)
    for which in ("row", "col"):
        if g[f"q_{which}"] is None:
            continue
        assert np.array_equal(gs[f"q_{which}"], g[f"q_{which}"])
        assert np.array_equal(gs[f"s_{which}"], relayout_tiled(g[f"s_{which}"]))


@pytest.mark.parametrize("scale", [1.75, 0.4])
def test_caller_supplied_amax_single_pass(scale):
    """Delayed scaling: nvfp4_quantize with an amax the caller supplies (here a
    previous step's value, larger or smaller than this tensor's own) and no
    amax pass.  A smaller amax saturates scale bytes at 448 and codes at the
    block maximum; GPU and oracle agree bit for bit either way, for the 1D, 4/6
    and 2D paths and with SR."""
    bits = small_input()
    x = to_device(bits)
    for flags, sel in ((ROW | COL, 0), (ROW | COL | F46, 1), (ROW | COL | TWO_D, 0), (ROW | COL | SR | F46, 2)):
        st, am = oracle.amax(bits, flags)
        supplied = (am * np.float32(scale)).astype(np.float32)
        g = gpu_quantize(x, flags, sel, sr_seed=9, amax=torch.from_numpy(supplied).cuda())
        r = oracle.quantize(bits, bits.shape[1], supplied, flags, sel=sel, sr_seed=9)
        r["amax"] = supplied
        assert_parity(g, r, flags)
        if scale < 1:
            assert (g["s_row"] == 0x7E).any()  # saturated scale bytes occur


@pytest.mark.parametrize("along_cols", [0, 1])
def test_transformed_values_agree_with_the_oracle(along_cols):
    """The tolerance on transformed values: the kernels' fp32 Hadamard
    transform (run alone through the test-only library, same device code) agrees with
    the oracle's (double precision, rounded once) within 1e-6 of each
    16-vector's 2-norm, for vectors along rows and along columns."""
    import ctypes
    f = selftest_lib().nvfp4_test_rht
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                  ctypes.c_void_p, ctypes.c_void_p]
    M, N, seed = 272, 528, 0xC0FFEE
    bits = small_input(M, N, kind="grad")
    x = to_device(bits)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert f(x.data_ptr(), M, N, N, along_cols, seed, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    g = out.cpu().numpy()
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    signs = oracle.rht_signs(seed)
    worst = 0.0
    if along_cols:
        vecs = [(slice(16 * b, 16 * b + 16), c) for b in range(M // 16) for c in range(N)]
    else:
        vecs = [(r, slice(16 * k, 16 * k + 16)) for r in range(M) for k in range(N // 16)]
    for idx in vecs:
        v = xf[idx]
        ref = oracle.rht16(v, signs)
        norm = float(np.linalg.norm(v.astype(np.float64)))
        err = float(np.abs(g[idx].astype(np.float64) - ref.astype(np.float64)).max())
        assert err <= 1e-6 * norm, (idx, err, norm)
        worst = max(worst, err / norm if norm else 0.0)
    assert worst < 1e-6


def test_scale_quotient_equals_ieee_division_exhaustively():
    """The kernels form each scale byte from a division-free quotient (a
    product and one residual correction).  For every finite bf16 block
    maximum b and every accepted bf16 amax A (b > A happens with a
    caller-supplied amax), for fp32 amax values between bf16 ones, and for 256
    random fp32 maxima per amax (Hadamard-transformed blocks), at Q = 6 over
    6*448 and Q = 6, 4 over 6*256, its E4M3 byte equals the byte of the IEEE
    quotient.  The bare product b * (1/den) does not have that property."""
    import ctypes
    f = selftest_lib().nvfp4_test_quotient_check
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    out = torch.zeros(6, dtype=torch.int64, device="cuda")
    assert f(out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    bytes_differ, _normal_quotients_differ, first, _quotients_differ, _two_steps, bare = out.tolist()
    assert bytes_differ == 0, hex(first)
    assert bare > 0  # the bare product b * (1/den) alone is not enough


def test_device_philox_equals_curand():
    """The kernels' Philox4x32-10 (stochastic-rounding words 0 and 1, RHT sign
    word) equals cuRAND's device implementation of the generator on 2^20
    counter/key cases, including every combination of extreme words; so do
    the form that takes the second-round product shared by one high word,
    and the 16-counter blocks the kernels draw (stride 1 and larger strides,
    some blocks crossing a multiple of 2^32)."""
    import ctypes
    hook = selftest_lib().nvfp4_test_philox_check
    hook.restype = ctypes.c_int
    hook.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    out = torch.zeros(6, dtype=torch.int64, device="cuda")
    assert hook(out.data_ptr(), 4096, None) == 0
    torch.cuda.synchronize()
    differ, differ_sign, checked, differ_shared, differ16, crossing = out.cpu().tolist()
    assert checked == 4096 * 256
    assert differ == 0 and differ_sign == 0
    assert differ_shared == 0 and differ16 == 0
    assert crossing > 100  # blocks of 16 counters across a multiple of 2^32 were among them


def _sr_cases(Q, rng):
    """Values and words for the stochastic rounding: random values on both
    sides of the grid and beyond Q, zeros, subnormals and tiny normals, and
    for values in every step region the words just below, at and above the
    decision boundary k = p * 2^24 (k = w >> 8, p the fraction of the step)."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    v = [rng.uniform(-8.0, 8.0, 40000), np.exp2(rng.uniform(-30, 3, 40000)) * rng.choice([-1.0, 1.0], 40000),
         np.array([0.0, -0.0, 2.0 ** -149, -(2.0 ** -149), 2.0 ** -126, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                   Q, -Q, Q + 0.25, 7.99, 100.0, -1e30]), grid, -grid, grid[1:] - 2.0 ** -20]
    v = np.concatenate(v).astype(np.float32)
    w = rng.integers(0, 2 ** 32, v.size, dtype=np.uint64).astype(np.uint32)
    # boundary words: m from each region, k in {ceil(P) - 1, ceil(P), floor(P)} with P = p * 2^24
    m = np.concatenate([rng.uniform(0.0, 0.5, 3000), rng.uniform(0.5, 1.0, 3000), rng.uniform(1.0, Q, 6000),
                        np.exp2(rng.uniform(-40, -1, 3000))]).astype(np.float32)
    bv, bw = [], []
    for mm in m.astype(np.float64):
        lo = grid[np.searchsorted(grid, mm, side="right") - 1]
        hi = grid[min(np.searchsorted(grid, mm, side="right"), grid.size - 1)]
        if hi == lo:
            continue
        P = (mm - lo) / (hi - lo) * 2.0 ** 24          # exact in double
        for k in {int(np.ceil(P)) - 1, int(np.ceil(P)), int(np.floor(P))}:
            if 0 <= k < 2 ** 24:
                bv.append(mm)
                bw.append((k << 8) | int(rng.integers(0, 256)))
    v = np.concatenate([v, np.array(bv, np.float32)])
    w = np.concatenate([w, np.array(bw, np.uint32)])
    return v, w


@pytest.mark.parametrize("Q", [6.0, 4.0])
def test_device_stochastic_rounding_equals_the_oracle(Q):
    """The kernels' stochastic rounding (run alone through the test-only
    library, same device code) gives the oracle's grid value, with the sign
    of the input, on random values, zeros, subnormals, values beyond Q, and
    words on both sides of and exactly at every decision boundary."""
    import ctypes
    hook = selftest_lib().nvfp4_test_sr_round
    hook.restype = ctypes.c_int
    hook.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                     ctypes.c_void_p]
    v, w = _sr_cases(Q, np.random.default_rng(20260 + int(Q)))
    vd = torch.from_numpy(v).cuda()
    wd = torch.from_numpy(w.view(np.int32)).cuda()
    out = torch.empty_like(vd)
    assert hook(vd.data_ptr(), wd.data_ptr(), v.size, Q, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    m = np.minimum(np.abs(v), np.float32(Q))
    ref = np.array([oracle.e2m1_value(oracle.round_sr(float(mm), int(ww))) for mm, ww in zip(m, w)], np.float32)
    ref = np.copysign(ref, v)
    bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert bad.size == 0, [(float(v[i]), hex(int(w[i])), float(got[i]), float(ref[i])) for i in bad[:5]]


@pytest.mark.parametrize("sr", [0, 1], ids=["rn", "sr"])
def test_tile_copy_timeout_is_reported_and_the_context_stays_usable(sr):
    """A 1D quantize kernel (round-to-nearest, or stochastic rounding on both
    copies) in a variant whose tile copies are never issued (test-only
    library: the barriers are armed, nothing arrives) stops after its bounded
    wait and reports NVFP4_ERR_PIPELINE in the status word; the next call on
    the same context is correct."""
    import ctypes
    hook = selftest_lib().nvfp4_test_quantize_no_copy
    hook.restype = ctypes.c_int
    hook.argtypes = ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 7 +
                     [ctypes.c_int, ctypes.c_void_p])
    flags = ROW | COL | (SR if sr else 0)
    M = 64
    bits = synthetic.weight(M, 256, 3)  # a single tile
    x = to_device(bits)
    amax = nv.nvfp4_amax(x, flags)
    out = nv.nvfp4_quantize(x, amax, flags)  # allocates the outputs
    out.status.zero_()
    torch.cuda.synchronize()
    p = lambda t: t.data_ptr()
    assert hook(p(x), M, 256, 256, p(amax), p(out.q_row), p(out.s_row), p(out.q_col), p(out.s_col), p(out.alpha),
                p(out.status), sr, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert out.status.item() == -8
    assert nv.nvfp4_strerror(-8).startswith("a tile copy")
    assert_parity(gpu_quantize(x, flags, sr_seed=5), ref_quantize(bits, flags, sr_seed=5), flags)


def test_two_d_copies_are_transposes_and_dequantize_identically():
    bits = synthetic.weight(256, 512, 17)
    for flags in (ROW | COL | TWO_D, ROW | COL | TWO_D | F46, ROW | COL | TWO_D | SR):
        g = gpu_quantize(to_device(bits), flags, 0, sr_seed=8)
        unpack = lambda q: np.stack([q & 15, q >> 4], -1).reshape(q.shape[0], -1)
        assert np.array_equal(unpack(g["q_col"]), unpack(g["q_row"]).T)
        out = g["_out"]
        dr = nv.nvfp4_dequantize(out.q_row, out.s_row, out.alpha[0:1])
        dc = nv.nvfp4_dequantize(out.q_col, out.s_col, out.alpha[1:2])
        assert torch.equal(dc.T.contiguous().view(torch.int32), dr.view(torch.int32))


@pytest.mark.parametrize("bf16", [False, True])
def test_dequantize_matches_oracle(bf16):
    bits = small_input()
    flags = ROW | COL | F46
    g = gpu_quantize(to_device(bits), flags, 0)
    out = g["_out"]
    for q, s, a, (rows, cols) in ((out.q_row, out.s_row, out.alpha[0:1], bits.shape),
                                  (out.q_col, out.s_col, out.alpha[1:2], bits.shape[::-1])):
        d = nv.nvfp4_dequantize(q, s, a, out_dtype=torch.bfloat16 if bf16 else torch.float32)
        torch.cuda.synchronize()
        ref = oracle.dequantize(q.cpu().numpy(), s.cpu().numpy(), float(a.item()), rows, cols, out_bf16=bf16)
        got = d.cpu().view(torch.int16 if bf16 else torch.int32).numpy()
        assert np.array_equal(got, ref.view(np.int16 if bf16 else np.int32))


def test_counter_offset_reproduces_a_row_shard():
    bits = synthetic.gradient(256, 512, 23)
    flags = ROW | COL | RHT_COL | SR
    x = to_device(bits)
    amax = nv.nvfp4_amax(x, flags, 77)
    whole = gpu_quantize(x, flags, 0, sr_seed=41, rht_seed=77, amax=amax)
    shard = gpu_quantize(x[128:], flags, 0, sr_seed=41, rht_seed=77, counter_offset=128 * 512, amax=amax)
    assert np.array_equal(shard["q_row"], whole["q_row"][128:])
    assert np.array_equal(shard["q_col"], whole["q_col"][:, 64:])
    assert np.array_equal(shard["s_col"], whole["s_col"][:, 8:])


@pytest.mark.parametrize("rht", [0, RHT_COL], ids=["plain", "rht_col"])
def test_both_copies_with_sr_equal_the_single_copy_kernels(rht):
    """With stochastic rounding on both copies, one Philox call per element
    serves both (word 0 rowwise, word 1 columnwise; the one-pass kernel rounds
    both in its columnwise pass).  Its rowwise copy equals what the
    rowwise-only kernel makes, and its columnwise copy what the
    columnwise-only kernel makes, from the same seeds and counters -- three
    code paths of the library that share no rounding loop."""
    bits = small_input(kind="grad")
    x = to_device(bits)
    kw = dict(sr_seed=0x77, rht_seed=0x99, counter_offset=(1 << 32) - 5000)
    both = gpu_quantize(x, ROW | COL | SR | rht, 0, **kw)
    row = gpu_quantize(x, ROW | SR, 0, **kw)
    col = gpu_quantize(x, COL | SR | rht, 0, **kw)
    assert np.array_equal(both["q_row"], row["q_row"]) and np.array_equal(both["s_row"], row["s_row"])
    assert np.array_equal(both["q_col"], col["q_col"]) and np.array_equal(both["s_col"], col["s_col"])


@pytest.mark.parametrize("offset", [(1 << 32) - 3000, (1 << 64) - 5000, (1 << 63) + 12345])
@pytest.mark.parametrize("flags", [ROW | COL | SR, ROW | COL | TWO_D | SR, ROW | COL | F46 | SR])
def test_counter_offsets_beyond_32_bits(offset, flags):
    """Philox counters (element index + offset, as a 64-bit integer) whose low
    word wraps inside the tensor, or whose 64-bit sum wraps, give the oracle's
    bits: the high counter word is carried and the sum is taken modulo 2^64."""
    bits = synthetic.activation_outlier_channels(128, 256, 61, frac=0.01)
    x = to_device(bits)
    g = gpu_quantize(x, flags, 0, sr_seed=0x5EEDF00D, counter_offset=offset)
    r = ref_quantize(bits.view(np.uint16), flags, 0, sr_seed=0x5EEDF00D, counter_offset=offset)
    assert_parity(g, r, flags)
    base = gpu_quantize(x, flags, 0, sr_seed=0x5EEDF00D, counter_offset=0)
    assert not np.array_equal(g["q_row"], base["q_row"])   # the offset reaches the rounding bits


def test_concurrent_host_threads_on_their_own_streams():
    """Several host threads, each on its own stream, quantize at once (the
    per-device launch caches are shared); every result equals the one-thread
    result."""
    import threading
    bits = small_input(M=384, N=768)
    x = to_device(bits)
    cases = [(ROW | COL | F46, 2), (ROW | COL | TWO_D | SR, 0), (ROW | COL | RHT_COL | SR | F46, 1),
             (COL | SR, 0), (ROW | RHT_ROW, 0), (ROW | COL | TWO_D | F46 | SR, 2)]
    want = [gpu_quantize(x, f, sel, sr_seed=9, rht_seed=10) for f, sel in cases]
    got = [None] * len(cases)
    errors = []

    def work(i):
        try:
            f, sel = cases[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(5):
                    amax = nv.nvfp4_amax(x, f, 10, stream=st)
                    out = nv.nvfp4_quantize(x, amax, f, sel, 9, 10, stream=st)
                st.synchronize()
            got[i] = out
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for w, g in zip(want, got):
        for k in ("q_row", "s_row", "q_col", "s_col"):
            t = getattr(g, k)
            if w[k] is None:
                assert t is None
            else:
                assert np.array_equal(t.cpu().numpy(), w[k]), k


def test_deterministic_and_graph_capturable():
    bits = small_input()
    flags = ROW | COL | RHT_COL | SR
    x = to_device(bits)
    a = gpu_quantize(x, flags, 0, sr_seed=3, rht_seed=4)
    b = gpu_quantize(x, flags, 0, sr_seed=3, rht_seed=4)
    for k in ("q_row", "s_row", "q_col", "s_col", "amax", "alpha"):
        assert np.array_equal(a[k], b[k])
    s = torch.cuda.Stream()
    amax = torch.empty(2, dtype=torch.float32, device="cuda")
    out = nv.nvfp4_quantize(x, a["_amax"], flags, 0, 3, 4)  # allocate outputs outside the capture
    torch.cuda.synchronize()
    for t in (out.q_row, out.q_col):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nv.nvfp4_amax(x, flags, 4, out=amax)
        nv.nvfp4_quantize(x, amax, flags, 0, 3, 4, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.q_row.cpu().numpy(), a["q_row"])
    assert np.array_equal(out.q_col.cpu().numpy(), a["q_col"])


# ------------------------------------------------------------------ full-size workloads
def assert_stripes_match_oracle(bits, g, flags, sel, stripes, sr_seed, rht_seed):
    """GPU outputs of a whole tensor against the oracle on 16-row stripes."""
    M, N = bits.shape
    st, am = oracle.amax(bits, flags, rht_seed)
    assert st == 0
    outs = oracle.output_buffers(M, N, flags)
    for sidx in stripes:
        oracle.quantize(bits, N, am, flags, sel=sel, sr_seed=sr_seed, rht_seed=rht_seed,
                        row0=16 * sidx, row1=16 * sidx + 16, outs=outs)
    q_row, s_row, q_col, s_col = outs
    rows = np.concatenate([np.arange(16 * s, 16 * s + 16) for s in stripes])
    pick = lambda d, qr, sr, qc, sc: dict(
        q_row=None if qr is None else qr[rows], s_row=None if sr is None else sr[rows],
        q_col=None if qc is None else np.concatenate([qc[:, 8 * s:8 * s + 8] for s in stripes], 1),
        s_col=None if sc is None else sc[:, stripes], **d)
    gs = pick(dict(amax=g["amax"], alpha=g["alpha"], status=g["status"]),
              g["q_row"], g["s_row"], g["q_col"], g["s_col"])
    alpha = (am / np.float32(1536.0 if flags & F46 else 2688.0)).astype(np.float32)
    rr = pick(dict(amax=am, alpha=alpha), q_row, s_row, q_col, s_col)
    assert_parity(gs, rr, flags)


@pytest.mark.parametrize("flags,sel", [(ROW | COL | SR, 0), (ROW | COL | F46, 1), (ROW | COL | TWO_D | F46 | SR, 0)])
def test_more_than_two_to_the_31_elements(flags, sel):
    """16400 x 131072 = 2.15e9 elements (4.3 GB of bf16): element indices,
    output offsets and Philox counters beyond 2^31, the tensor maximum in the
    last rows; stripes at both ends and across the 2^31 boundary are compared
    with the oracle exactly."""
    M, N = 16400, 131072
    bits = synthetic.tiled_large(M, N, 77)
    x = to_device(bits)
    g = gpu_quantize(x, flags, sel, sr_seed=0xABCDEF, rht_seed=0)
    del x
    torch.cuda.empty_cache()
    boundary = (1 << 31) // N // 16          # the stripe holding element 2^31
    stripes = sorted(s for s in {0, 1, boundary - 1, boundary, boundary + 1, M // 16 - 1} if s < M // 16)
    assert_stripes_match_oracle(bits, g, flags, sel, stripes, 0xABCDEF, 0)
    assert float(g["amax"][0]) == 56.0


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_workload_full_size_every_element(name):
    """Each workload of the recipe at its full size, in the launch
    configuration the benchmark times: every code and scale byte of both
    copies equals the oracle's (within the Hadamard tolerance over the whole
    tensor for a transformed copy).  The oracle runs on every host core."""
    from oracle.parallel import quantize_parallel
    flags, sel = synthetic.workload_flags(name)
    bits = synthetic.workload(name)
    x = to_device(bits)
    g = gpu_quantize(x, flags, sel, sr_seed=synthetic.SR_SEED, rht_seed=synthetic.RHT_SEED)
    del x
    torch.cuda.empty_cache()
    r = quantize_parallel(bits, flags, sel, sr_seed=synthetic.SR_SEED, rht_seed=synthetic.RHT_SEED)
    assert r["status"] == 0
    assert_parity(g, r, flags)


@pytest.mark.parametrize("flags,sel", [(ROW | COL | SR, 0), (ROW | COL | RHT_COL | SR, 0), (ROW | COL | TWO_D, 0),
                                       (ROW | COL | F46, 1), (ROW | COL | TWO_D | SR | F46, 2)])
def test_row_sharded_recipe_through_the_library(flags, sel):
    """The multi-GPU recipe, run through the library on one GPU: the tensor
    is split into two row stripes (multiples of 16 rows); each stripe's amax
    comes from its own nvfp4_amax call, the host takes the MAX of the stripes'
    values (the all-reduce), and each stripe is quantized with that amax and
    counter_offset = first_row * N.  The gathered outputs equal the unsharded
    call bit for bit (SR words included)."""
    M, N, split = 320, 528, 144
    bits = synthetic.gradient(M, N, 29) if flags & (SR | RHT_COL) else small_input(M, N)
    x = to_device(bits)
    whole = gpu_quantize(x, flags, sel, sr_seed=0x77, rht_seed=0x99)
    parts = [(0, split), (split, M)]
    amaxes = [nv.nvfp4_amax(x[r0:r1], flags, 0x99) for r0, r1 in parts]
    am = torch.maximum(amaxes[0], amaxes[1])  # the MAX all-reduce of two float pairs
    shards = [gpu_quantize(x[r0:r1], flags, sel, sr_seed=0x77, rht_seed=0x99, counter_offset=r0 * N, amax=am)
              for r0, r1 in parts]
    assert np.array_equal(am.cpu().numpy(), whole["amax"])
    for sh in shards:
        assert np.array_equal(sh["alpha"], whole["alpha"])
    assert np.array_equal(np.concatenate([s["q_row"] for s in shards]), whole["q_row"])
    assert np.array_equal(np.concatenate([s["s_row"] for s in shards]), whole["s_row"])
    assert np.array_equal(np.concatenate([s["q_col"] for s in shards], 1), whole["q_col"])
    assert np.array_equal(np.concatenate([s["s_col"] for s in shards], 1), whole["s_col"])
