"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and rounds them to bfloat16; it holds
none of the quantizer's arithmetic, and neither the CUDA path nor the oracle
imports the other through it.  Every tensor is returned as a numpy ``uint16``
array of bfloat16 bit patterns (row-major, M x N), drawn with numpy's PCG64 in
row chunks and rounded to bfloat16 (nearest even) by torch on the CPU.

Workloads (shapes and value distributions of the NVFP4 training recipe):

* ``activation_outlier_entries``: N(0,1), a fraction of entries at seeded
  positions scaled by a factor (1x16 rowwise case, 256 x 1024, 0.1%, x50);
* ``activation_outlier_channels``: N(0,1), a fraction of whole columns
  (hidden channels) scaled (8192 x 5120, 0.05%, x30);
* ``weight``: N(0, 0.02) (5120 x 20480);
* ``gradient``: Student-t with 3 degrees of freedom scaled by 1e-3
  (16384 x 5120, and 16384 x 20480 for dY).
"""
from __future__ import annotations

import numpy as np
import torch

DATA_SEED_BASE = 20251202
_CHUNK_ROWS = 1024


def _to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _fill(M: int, N: int, rng: np.random.Generator, draw) -> np.ndarray:
    out = np.empty((M, N), dtype=np.uint16)
    for r0 in range(0, M, _CHUNK_ROWS):
        r1 = min(M, r0 + _CHUNK_ROWS)
        out[r0:r1] = _to_bf16_bits(draw(rng, (r1 - r0, N)))
    return out


def activation_outlier_entries(M: int, N: int, seed: int, frac: float = 0.001,
                               scale: float = 50.0) -> np.ndarray:
    """N(0,1) with round(frac*M*N) distinct seeded positions multiplied by ``scale``."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N), dtype=np.float32)
    k = int(round(frac * M * N))
    pos = rng.permutation(M * N)[:k]
    x.reshape(-1)[pos] *= np.float32(scale)
    return _to_bf16_bits(x)


def activation_outlier_channels(M: int, N: int, seed: int, frac: float = 0.0005,
                                scale: float = 30.0) -> np.ndarray:
    """N(0,1) with max(1, round(frac*N)) seeded columns multiplied by ``scale``."""
    rng = np.random.default_rng(seed)
    k = max(1, int(round(frac * N)))
    cols = np.sort(rng.permutation(N)[:k])
    mult = np.ones(N, dtype=np.float32)
    mult[cols] = np.float32(scale)
    return _fill(M, N, rng, lambda g, shape: g.standard_normal(shape, dtype=np.float32) * mult)


def weight(M: int, N: int, seed: int, std: float = 0.02) -> np.ndarray:
    """N(0, std^2)."""
    rng = np.random.default_rng(seed)
    return _fill(M, N, rng, lambda g, shape: g.standard_normal(shape, dtype=np.float32) * np.float32(std))


def gradient(M: int, N: int, seed: int, nu: float = 3.0, scale: float = 1e-3) -> np.ndarray:
    """Student-t(nu) * scale (heavy-tailed, like wgrad operands)."""
    rng = np.random.default_rng(seed)
    return _fill(M, N, rng, lambda g, shape: (g.standard_t(nu, shape) * scale).astype(np.float32))


# The workloads of the recipe: name -> (generator, M, N, seed, flags, selection rule).
# flags: 1 rowwise, 2 columnwise, 4 2D, 16 Hadamard on the columnwise copy,
# 32 stochastic rounding, 64 4/6; selection 0 MAE, 1 MSE.
WORKLOADS = {
    "rowwise_rn_256x1024": (activation_outlier_entries, 256, 1024, DATA_SEED_BASE + 1, 1, 0),
    "act_46mae_8192x5120": (activation_outlier_channels, 8192, 5120, DATA_SEED_BASE + 2, 1 | 2 | 64, 0),
    "weight_2d_5120x20480": (weight, 5120, 20480, DATA_SEED_BASE + 3, 1 | 2 | 4, 0),
    "grad_rht_sr_16384x5120": (gradient, 16384, 5120, DATA_SEED_BASE + 4, 1 | 2 | 16 | 32, 0),
    "linear_x_16384x5120": (activation_outlier_channels, 16384, 5120, DATA_SEED_BASE + 5, 1 | 2 | 64, 1),
    "linear_w_5120x20480": (weight, 5120, 20480, DATA_SEED_BASE + 6, 1 | 2 | 4, 0),
    "linear_dy_16384x20480": (gradient, 16384, 20480, DATA_SEED_BASE + 7, 1 | 2 | 16 | 32, 0),
}
SR_SEED = 0x1234ABCD
RHT_SEED = 0x5EED


def workload(name: str, M: int | None = None, N: int | None = None) -> np.ndarray:
    """The named workload's distribution at its own size, or at (M, N)."""
    gen, M0, N0, seed = WORKLOADS[name][:4]
    return gen(M or M0, N or N0, seed)


def tiled_large(M: int, N: int, seed: int, block_rows: int = 256) -> np.ndarray:
    """A tensor too large to draw element by element in a test: a seeded
    N(0,1) block of ``block_rows`` x N rows with outlier channels, repeated down
    the rows, plus three seeded entries set to 40, 48 and 56 in the last rows
    (so the tensor maximum lies beyond the first 2^31 elements)."""
    block = activation_outlier_channels(block_rows, N, seed, frac=0.001, scale=8.0)
    out = np.empty((M, N), dtype=np.uint16)
    for r0 in range(0, M, block_rows):
        r1 = min(M, r0 + block_rows)
        out[r0:r1] = block[:r1 - r0]
    rng = np.random.default_rng(seed + 1)
    for v in (40.0, 48.0, 56.0):
        r = int(rng.integers(max(0, M - 16), M))
        c = int(rng.integers(0, N))
        out[r, c] = _to_bf16_bits(np.array([v], np.float32))[0]
    return out


def workload_flags(name: str):
    """(flags, selection rule) of the named workload."""
    return WORKLOADS[name][4], WORKLOADS[name][5]
