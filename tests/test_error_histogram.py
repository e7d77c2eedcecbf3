"""The quantization-error histogram (oracle side, CPU).

The oracle's histogram is pinned against an independent numpy restatement of
its definition on seeded tensors, against invariants, and against the 4/6
page's worked example (Problem statement): a value at 75 % of its block
maximum sits at scaled value 4.5 when the block is scaled to 6 -- in the gap
between 4 and 6, rounding error 0.5 -- and exactly on "3" when it is scaled
to 4 (error 0).
"""
import numpy as np
import pytest

import oracle
import synthetic

ROW, F46 = 1, 64
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def e4m3_values():
    """Every E4M3 byte's value from its definition (bias 7, subnormal step 2^-9)."""
    out = np.zeros(256, np.float32)
    for e in range(256):
        exp, man = (e >> 3) & 15, e & 7
        mag = man * 2.0 ** -9 if exp == 0 else (1 + man / 8) * 2.0 ** (exp - 7)
        out[e] = -mag if e & 128 else mag
    return out


def numpy_histogram(bits, q, s, alpha, nbins):
    """The histogram's definition restated with numpy float32 operations."""
    x = bf16_to_f32(bits)
    M, N = x.shape
    codes = np.stack([q & 15, q >> 4], -1).reshape(M, N)
    val = np.where(codes & 8, -GRID[codes & 7], GRID[codes & 7]).astype(np.float32)
    d = (e4m3_values()[s] * np.float32(alpha)).astype(np.float32)       # M x N/16
    xh = (val * np.repeat(d, 16, axis=1)).astype(np.float32)
    b = np.abs(x).reshape(M, N // 16, 16).max(-1)
    bb = np.repeat(b, 16, axis=1)
    keep = bb > 0
    f6, fnb = np.float32(6), np.float32(nbins)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (f6 * np.abs(x)).astype(np.float32) / bb
        binf = np.floor(((v * fnb).astype(np.float32) / f6).astype(np.float32))
        e = ((f6 * np.abs((x - xh).astype(np.float32))).astype(np.float32) / bb).astype(np.float32)
    bins = np.minimum(binf[keep].astype(np.int64), nbins - 1)
    e = e[keep]
    e24 = (e * np.float32(2 ** 24)).astype(np.float32).astype(np.uint64)
    ee32 = ((e * e).astype(np.float32) * np.float32(2 ** 32)).astype(np.float32).astype(np.uint64)
    hist = np.zeros((3, nbins), np.uint64)
    np.add.at(hist[0], bins, 1)
    np.add.at(hist[1], bins, e24)
    np.add.at(hist[2], bins, ee32)
    return hist


def quantized(bits, flags, sel=0):
    st, am = oracle.amax(bits, flags)
    r = oracle.quantize(bits, bits.shape[1], am, flags, sel=sel)
    return r["q_row"], r["s_row"], float(r["alpha"][0])


@pytest.mark.parametrize("flags,sel,nbins", [(ROW, 0, 24), (ROW | F46, 0, 24), (ROW | F46, 1, 7), (ROW, 0, 1)])
def test_oracle_histogram_equals_numpy_restatement(flags, sel, nbins):
    bits = synthetic.activation_outlier_channels(48, 256, 3, frac=0.02).view(np.uint16).copy()
    bits[5, 16:32] = 0                     # a zero block is skipped
    q, s, alpha = quantized(bits, flags, sel)
    got = oracle.error_histogram(bits, 256, q, s, alpha, nbins)
    assert np.array_equal(got, numpy_histogram(bits, q, s, alpha, nbins))
    assert int(got[0].sum()) == 48 * 256 - 16
    # the block maxima (v = 6) land in the last bin
    assert int(got[0, -1]) >= 48 * 256 // 16 - 1


def test_page_example_seventy_five_percent_of_the_max():
    b = np.float32(2.625)                   # 2688 * 2^-10: d = b/6 exactly at scale 6, b/4 at scale 4
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1] = b, np.float32(0.75) * b
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_to_f32(bits), x)
    std = oracle.error_histogram(bits, 16, *quantized(bits, ROW), nbins=24)
    four = oracle.error_histogram(bits, 16, *quantized(bits, ROW | F46), nbins=24)
    assert std[0].tolist() == four[0].tolist() == [14] + [0] * 17 + [1] + [0] * 4 + [1]
    assert int(std[1, 18]) == 2 ** 23 and int(std[2, 18]) == 2 ** 30   # e = 0.5 in the 4-6 gap at scale 6
    assert int(four[1].sum()) == 0 and int(four[2].sum()) == 0          # exactly "3" and "4" at scale 4
