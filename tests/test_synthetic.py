"""The seeded input generators: deterministic, the documented shapes and
distributions, and bfloat16 rounding to nearest even."""
import numpy as np
import pytest
import torch

import synthetic


def f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_same_seed_same_bits_other_seed_other_bits():
    a = synthetic.activation_outlier_channels(64, 256, 5)
    b = synthetic.activation_outlier_channels(64, 256, 5)
    c = synthetic.activation_outlier_channels(64, 256, 6)
    assert a.dtype == np.uint16 and a.shape == (64, 256)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_chunked_draw_equals_one_draw():
    """Rows are drawn in chunks; a tensor taller than one chunk equals the
    same draws made in one piece (rounded to bfloat16 the same way)."""
    M, N, seed = synthetic._CHUNK_ROWS + 40, 64, 11
    got = synthetic.weight(M, N, seed)
    rng = np.random.default_rng(seed)
    parts = []
    for r0 in range(0, M, synthetic._CHUNK_ROWS):
        n = min(M, r0 + synthetic._CHUNK_ROWS) - r0
        parts.append(rng.standard_normal((n, N), dtype=np.float32) * np.float32(0.02))
    want = torch.from_numpy(np.concatenate(parts)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to the even mantissa (1.0);
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)], np.float32)
    got = f32(synthetic._to_bf16_bits(x))
    assert got.tolist() == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0]


def test_outlier_channels_are_whole_columns():
    bits = synthetic.activation_outlier_channels(512, 2048, 3, frac=0.002, scale=30.0)
    x = f32(bits)
    col_rms = np.sqrt((x.astype(np.float64) ** 2).mean(0))
    k = max(1, int(round(0.002 * 2048)))
    hot = np.argsort(col_rms)[-k:]
    assert np.all(col_rms[hot] > 20) and np.all(np.delete(col_rms, hot) < 1.2)


def test_outlier_entries_count():
    bits = synthetic.activation_outlier_entries(256, 1024, 9, frac=0.001, scale=50.0)
    x = np.abs(f32(bits))
    # N(0,1) entries beyond 10 essentially never occur; scaled entries mostly do
    n_big = int((x > 10).sum())
    assert 0.8 * 262 <= n_big <= 262


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_workload_shapes_and_flags(name):
    gen, M, N, seed, flags, sel = synthetic.WORKLOADS[name]
    assert M % 16 == 0 and N % 16 == 0 and flags & 3 and sel in (0, 1, 2)
    assert synthetic.workload_flags(name) == (flags, sel)
    small = synthetic.workload(name, 32, 64)
    assert small.shape == (32, 64) and np.isfinite(f32(small)).all()


def test_tiled_large_repeats_its_block_and_plants_the_maximum():
    M, N = 600, 128
    t = synthetic.tiled_large(M, N, 4, block_rows=256)
    block = synthetic.activation_outlier_channels(256, N, 4, frac=0.001, scale=8.0)
    assert np.array_equal(t[:256], block) and np.array_equal(t[256:512], block)
    x = np.abs(f32(t))
    assert x.max() == 56.0 and np.argmax(x) // N >= M - 16
