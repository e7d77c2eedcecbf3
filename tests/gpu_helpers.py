"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding, run the oracle on the same seeded input, and compare.

Bar (the method's stated tolerances):
* no Hadamard transform on a copy: amax, alpha, every code byte and every scale
  byte bit-exact;
* Hadamard-transformed copy: amax and alpha within 1e-6 relative; at most
  0.01 % of codes differ, each by at most one signed grid step (+-0 equal);
  at most 0.01 % of scale bytes differ, each by at most one E4M3 step.

Every output buffer the GPU path writes is surrounded by guard bytes holding
a canary value, and in the tiled scale layout the padding entries hold it too;
after each call the canaries must be intact, so a store past a row, a tile
edge or the end of a buffer fails the test.
"""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_bit_block_gb300 as nv
import oracle

RHT_CODE_FRAC = 1e-4
RHT_REL = 1e-6


def to_device(bits: np.ndarray, ld: int | None = None) -> torch.Tensor:
    """bf16 bit patterns (M x N uint16) -> CUDA bf16 tensor, optionally with
    a padded row stride ld >= N (a column slice of a wider buffer)."""
    M, N = bits.shape
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if ld is None or ld == N:
        return t.cuda()
    wide = torch.zeros((M, ld), dtype=torch.bfloat16)
    wide[:, :N] = t
    return wide.cuda()[:, :N]


GUARD = 512          # guard bytes before and after every output buffer
CANARY = 0xA5


class Guarded:
    """A uint8 CUDA buffer of `shape` inside a larger one whose guard bytes
    (and, for a tiled scale buffer, the padding entries) hold CANARY."""

    def __init__(self, shape, pad_mask=None):
        n = int(np.prod(shape))
        self.base = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.view = self.base[GUARD:GUARD + n].view(shape)
        self.pad_mask = pad_mask  # bool array of `shape`: entries the kernel must not write

    def check(self, what: str):
        h = self.base.cpu().numpy()
        n = h.size - 2 * GUARD
        assert (h[:GUARD] == CANARY).all(), f"{what}: bytes written before the buffer"
        assert (h[GUARD + n:] == CANARY).all(), f"{what}: bytes written after the buffer"
        if self.pad_mask is not None:
            body = h[GUARD:GUARD + n].reshape(self.view.shape)
            assert (body[self.pad_mask] == CANARY).all(), f"{what}: padding entries of the tiled layout written"


def tiled_padding_mask(R: int, C: int) -> np.ndarray:
    """Entries of the tiled scale layout (rows padded to 128, scale columns to
    4) that hold no scale: the layout's definition restated (128 x 4 tiles of
    512 bytes, scale (r, c) at (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4)."""
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    used = np.zeros(Rp * Cp, bool)
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    used[((r // 128) * (Cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4] = True
    return ~used.reshape(Rp, Cp)


def guarded_outputs(M: int, N: int, flags: int):
    """Quantized(...) whose code and scale buffers are Guarded; returns (out, guards)."""
    shapes = nv.output_shapes(M, N, flags)
    swz = bool(flags & nv.SF_SWIZZLED)
    guards = {}
    views = []
    for name, shp in zip(("q_row", "s_row", "q_col", "s_col"), shapes):
        if shp is None:
            views.append(None)
            continue
        mask = None
        if swz and name.startswith("s_"):
            R, C = (M, N // 16) if name == "s_row" else (N, M // 16)
            mask = tiled_padding_mask(R, C)
        g = Guarded(shp, mask)
        guards[name] = g
        views.append(g.view)
    out = nv.Quantized(*views, alpha=torch.empty(2, dtype=torch.float32, device="cuda"),
                       status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return out, guards


def gpu_quantize(x: torch.Tensor, flags: int, sel: int = 0, sr_seed: int = 0, rht_seed: int = 0,
                 counter_offset: int = 0, amax=None):
    """The CUDA path through the C ABI, with guarded outputs whose canaries
    are checked after the call."""
    if amax is None:
        amax = nv.nvfp4_amax(x, flags, rht_seed)
    out, guards = guarded_outputs(x.shape[0], x.shape[1], flags)
    nv.nvfp4_quantize(x, amax, flags, sel, sr_seed, rht_seed, counter_offset, out=out)
    torch.cuda.synchronize()
    for name, g in guards.items():
        g.check(name)
    host = lambda t: None if t is None else t.cpu().numpy()
    res = dict(amax=host(amax), alpha=host(out.alpha), status=int(out.status.item()),
               q_row=host(out.q_row), s_row=host(out.s_row), q_col=host(out.q_col), s_col=host(out.s_col),
               _out=out, _amax=amax)
    if flags & nv.SF_SWIZZLED:  # the padding holds the canary; report it as zero like a zeroed buffer
        for name, g in guards.items():
            if g.pad_mask is not None:
                res[name] = np.where(g.pad_mask, 0, res[name]).astype(np.uint8)
    return res


_selftest = None


def selftest_lib():
    """The test-only self-check library (tests/selftest), built on first use."""
    global _selftest
    if _selftest is None:
        import ctypes
        from nvfp4_bit_block_gb300.build import build_selftest
        _selftest = ctypes.CDLL(build_selftest())
    return _selftest


def ref_quantize(bits: np.ndarray, flags: int, sel: int = 0, sr_seed: int = 0, rht_seed: int = 0,
                 counter_offset: int = 0):
    M, N = bits.shape
    st, am = oracle.amax(bits, flags, rht_seed)
    assert st == 0
    out = oracle.quantize(bits, N, am, flags, sel=sel, sr_seed=sr_seed, rht_seed=rht_seed,
                          counter_offset=counter_offset)
    out["amax"] = am
    return out


def signed_grid_index(q: np.ndarray) -> np.ndarray:
    codes = np.stack([q & 15, q >> 4], -1).reshape(q.shape[0], -1).astype(np.int16)
    mag = codes & 7
    return np.where(codes & 8, -mag, mag)


def _first_diff(a, b):
    idx = np.argwhere(a != b)
    return f"{len(idx)} differ, first at {tuple(idx[0])}: gpu {a[tuple(idx[0])]} ref {b[tuple(idx[0])]}"


def assert_copy_exact(g, r, which: str):
    q, s = f"q_{which}", f"s_{which}"
    assert np.array_equal(g[s], r[s]), f"{s}: " + _first_diff(g[s], r[s])
    assert np.array_equal(g[q], r[q]), f"{q}: " + _first_diff(g[q], r[q])


def assert_copy_close(g, r, which: str):
    q, s = f"q_{which}", f"s_{which}"
    dg, dr = signed_grid_index(g[q]), signed_grid_index(r[q])
    dq = np.abs(dg - dr)
    assert dq.max(initial=0) <= 1, f"{q}: a code differs by {dq.max()} steps"
    assert (dq != 0).mean() <= RHT_CODE_FRAC, f"{q}: {(dq != 0).mean():.2e} of codes differ"
    ds = np.abs(g[s].astype(np.int16) - r[s].astype(np.int16))
    assert ds.max(initial=0) <= 1, f"{s}: a scale differs by {ds.max()} steps"
    assert (ds != 0).mean() <= RHT_CODE_FRAC, f"{s}: {(ds != 0).mean():.2e} of scales differ"


def assert_scalar(gv, rv, exact: bool, what: str):
    gv, rv = np.float32(gv), np.float32(rv)
    if exact:
        assert gv.view(np.uint32) == rv.view(np.uint32), f"{what}: gpu {gv!r} ref {rv!r}"
    else:
        assert abs(float(gv) - float(rv)) <= RHT_REL * abs(float(rv)), f"{what}: gpu {gv!r} ref {rv!r}"


def assert_parity(g, r, flags: int):
    row_exact = not flags & nv.RHT_ROW
    col_exact = not flags & nv.RHT_COL
    assert g["status"] == 0
    if flags & nv.ROWWISE:
        assert_scalar(g["amax"][0], r["amax"][0], row_exact, "amax[0]")
        assert_scalar(g["alpha"][0], r["alpha"][0], row_exact, "alpha[0]")
        (assert_copy_exact if row_exact else assert_copy_close)(g, r, "row")
    if flags & nv.COLWISE:
        assert_scalar(g["amax"][1], r["amax"][1], col_exact, "amax[1]")
        assert_scalar(g["alpha"][1], r["alpha"][1], col_exact, "alpha[1]")
        (assert_copy_exact if col_exact else assert_copy_close)(g, r, "col")
