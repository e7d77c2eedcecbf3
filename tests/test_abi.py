"""The C-ABI library loads, exports what include/nvfp4.h declares, and rejects
bad arguments on the host (no GPU needed: these calls return before any CUDA
work is enqueued)."""
import ctypes
import os
import re
import subprocess

import pytest

import nvfp4_bit_block_gb300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")

ALIGNED = 0x100000       # fake, 16-byte aligned "device" addresses: never dereferenced
ALIGNED2 = 0x200000
ALIGNED3 = 0x300000


@pytest.fixture(scope="module")
def L():
    nv.build()
    return nv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*NVFP4_API\s+(?:int|const char\*)\s+(nvfp4_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == ["nvfp4_amax", "nvfp4_dequantize", "nvfp4_error_histogram", "nvfp4_gemm",
                                    "nvfp4_quantize", "nvfp4_strerror"]


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", nv.build()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (nvfp4_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_library_is_built_for_sm_103a_only():
    out = subprocess.run(["/usr/local/cuda/bin/cuobjdump", "--list-elf", nv.build()], capture_output=True,
                         text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    arches = set(re.findall(r"sm_(\d+a?)", out.stdout))
    assert arches == {"103a"}, arches


def test_strerror(L):
    assert nv.nvfp4_strerror(0) == "ok"
    for st in (-1, -2, -3, -4, -5, -6, -7, -8):
        assert nv.nvfp4_strerror(st) not in ("", "unknown status")
    assert nv.nvfp4_strerror(12345) == "unknown status"


def quantize(L, x=ALIGNED, M=32, N=32, ld=32, amax=ALIGNED2, flags=3, sel=0,
             q_row=ALIGNED, s_row=ALIGNED, q_col=ALIGNED, s_col=ALIGNED, alpha=ALIGNED3, status=None):
    return L.nvfp4_quantize(x, M, N, ld, amax, flags, sel, 0, 0, 0, q_row, s_row, q_col, s_col, alpha,
                            status, None)


def test_quantize_rejects_bad_arguments(L):
    assert quantize(L, flags=0) == -4                          # no copy requested
    assert quantize(L, flags=3 | 256) == -4                    # unknown bit
    assert quantize(L, flags=3 | 4 | 8) == -4                  # 2D with an RHT flag
    assert quantize(L, flags=2 | 8) == -4                      # row RHT without the row copy
    assert quantize(L, flags=1 | 16) == -4                     # col RHT without the col copy
    assert quantize(L, flags=3 | 64, sel=3) == -4              # selection rule out of range
    assert quantize(L, N=24, ld=24) == -2                      # N % 16
    assert quantize(L, M=24) == -2                             # M % 16 with COLWISE
    assert quantize(L, M=-16) == -2
    assert quantize(L, ld=16) == -2                            # ld < N
    assert quantize(L, N=32, ld=36) == -3                      # ld % 8
    assert quantize(L, x=ALIGNED + 8) == -3                    # x not 16-byte aligned
    assert quantize(L, q_row=ALIGNED + 4) == -3
    assert quantize(L, s_col=ALIGNED + 1) == -3
    assert quantize(L, amax=None) == -1
    assert quantize(L, alpha=None) == -1
    assert quantize(L, x=None) == -1
    assert quantize(L, q_col=None) == -1
    assert quantize(L, flags=1, q_col=None, s_col=None) != -1  # not needed without COLWISE
    assert quantize(L, M=2 ** 31, N=32, flags=1) == -2         # beyond 32-bit tile coordinates


def test_amax_and_dequantize_reject_bad_arguments(L):
    assert L.nvfp4_amax(ALIGNED, 32, 24, 24, 1, 0, ALIGNED2, None) == -2
    assert L.nvfp4_amax(ALIGNED, 32, 32, 32, 0, 0, ALIGNED2, None) == -4
    assert L.nvfp4_amax(ALIGNED, 32, 32, 32, 1, 0, None, None) == -1
    assert L.nvfp4_amax(ALIGNED + 2, 32, 32, 32, 1, 0, ALIGNED2, None) == -3
    assert L.nvfp4_dequantize(ALIGNED, ALIGNED, ALIGNED2, 4, 24, 0, ALIGNED3, None) == -2
    assert L.nvfp4_dequantize(None, ALIGNED, ALIGNED2, 4, 32, 0, ALIGNED3, None) == -1
    assert L.nvfp4_dequantize(ALIGNED, ALIGNED, ALIGNED2, 4, 32, 0, ALIGNED3 + 8, None) == -3
    assert L.nvfp4_dequantize(ALIGNED, ALIGNED, ALIGNED2, 0, 32, 0, ALIGNED3, None) == 0  # empty: no-op


def _has_gpu():
    import torch
    return torch.cuda.is_available()


def test_launch_failure_is_reported(L):
    """On a machine without a GPU, calls that pass the host-side checks fail
    in the CUDA runtime before anything runs, and report NVFP4_ERR_CUDA.
    (Skipped where a GPU is present: the fake addresses would reach a kernel.)"""
    if _has_gpu():
        pytest.skip("needs a machine without a GPU: the fake device addresses would be launched")
    assert quantize(L) == -5
    assert L.nvfp4_amax(ALIGNED, 32, 32, 32, 1, 0, ALIGNED2, None) == -5
    assert L.nvfp4_dequantize(ALIGNED, ALIGNED, ALIGNED2, 4, 32, 0, ALIGNED3, None) == -5


def test_product_library_exports_no_test_hooks():
    """The self-checks live in the test-only library; the product library
    exports exactly the entry points of include/nvfp4.h."""
    out = subprocess.run(["nm", "-D", "--defined-only", nv.build()], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r"\bT (nvfp4_\w+)", out)))
    assert exported == declared_functions()


def test_binding_raises_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nv, "_lib", None)
    monkeypatch.setattr(nv, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        nv.lib()


def test_gemm_rejects_bad_arguments(L):
    g = L.nvfp4_gemm
    g.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                                                  ctypes.c_void_p, ctypes.c_void_p]
    ok = [ALIGNED, ALIGNED, ALIGNED2, ALIGNED, ALIGNED, ALIGNED2, 128, 128, 256, 0, ALIGNED3, 128, None, None]
    call = lambda changes: g(*[changes.get(i, v) for i, v in enumerate(ok)])
    assert call({6: 100}) == -2 and call({7: 200}) == -2 and call({8: 128}) == -2   # M, N % 128; K % 256
    assert call({8: 0}) == -2 and call({11: 64}) == -2                             # K = 0; ldd < N
    assert call({6: 0}) == 0                                                       # empty: no-op
    assert call({0: None}) == -1 and call({2: None}) == -1 and call({10: None}) == -1
    assert call({0: ALIGNED + 8}) == -3 and call({1: ALIGNED + 4}) == -3           # codes, scales 16-byte
    assert call({10: ALIGNED3 + 4}) == -3 and call({11: 130}) == -3                # D 16-byte, ldd % 4
    assert call({9: 1, 11: 132}) == -3                                             # bf16 rows: ldd % 8


def test_error_histogram_rejects_bad_arguments(L):
    h = L.nvfp4_error_histogram
    h.restype = ctypes.c_int
    h.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    ok = dict(x=ALIGNED, M=32, N=32, ld=32, q=ALIGNED, s=ALIGNED, a=ALIGNED2, nb=24, hist=ALIGNED3)

    def call(**kw):
        d = dict(ok, **kw)
        return h(d["x"], d["M"], d["N"], d["ld"], d["q"], d["s"], d["a"], d["nb"], d["hist"], None)
    assert call(N=40) == -2 and call(ld=16) == -2 and call(nb=0) == -2 and call(nb=1025) == -2
    assert call(hist=None) == -1 and call(q=None) == -1
    assert call(x=ALIGNED + 8) == -3 and call(ld=36) == -3
    assert call(M=0) == 0


def test_binding_has_the_c_names():
    for name in ("nvfp4_amax", "nvfp4_quantize", "nvfp4_dequantize", "nvfp4_error_histogram", "nvfp4_strerror"):
        assert callable(getattr(nv, name))


def test_binding_rejects_host_tensors_before_any_launch():
    """Host (CPU) tensors never reach the library: their addresses would be
    dereferenced on the GPU."""
    import torch
    x = torch.zeros((32, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        nv.nvfp4_amax(x, 3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        nv.nvfp4_quantize(x, torch.zeros(2), 3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        nv.nvfp4_error_histogram(x, None, None, None)
    with pytest.raises(ValueError, match="CUDA tensor"):
        nv.nvfp4_dequantize(torch.zeros((16, 8), dtype=torch.uint8), torch.zeros((16, 1), dtype=torch.uint8),
                            torch.zeros(1))
    with pytest.raises(TypeError):
        nv.nvfp4_amax(torch.zeros((32, 32), dtype=torch.float32), 3)


def test_self_check_hooks_reject_bad_arguments():
    """The GPU self-check hooks (test-only library) validate on the host
    before launching."""
    from nvfp4_bit_block_gb300.build import build_selftest
    L = ctypes.CDLL(build_selftest())
    ph = L.nvfp4_test_philox_check
    ph.restype = ctypes.c_int
    ph.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert ph(None, 16, None) == -1 and ph(ALIGNED, 0, None) == -2 and ph(ALIGNED, -3, None) == -2
    qc = L.nvfp4_test_quotient_check
    qc.restype = ctypes.c_int
    qc.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert qc(None, None) == -1
    rh = L.nvfp4_test_rht
    rh.restype = ctypes.c_int
    rh.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                   ctypes.c_void_p, ctypes.c_void_p]
    assert rh(None, 16, 16, 16, 0, 0, ALIGNED, None) == -1
    assert rh(ALIGNED, 16, 24, 24, 0, 0, ALIGNED2, None) == -2      # N % 16
    assert rh(ALIGNED, 24, 16, 16, 1, 0, ALIGNED2, None) == -2      # along columns needs M % 16
    assert rh(ALIGNED, 16, 16, 8, 0, 0, ALIGNED2, None) == -2       # ld < N
    assert rh(ALIGNED + 2, 16, 16, 16, 0, 0, ALIGNED2, None) == -3  # x not 4-byte aligned
    assert rh(ALIGNED, 16, 16, 17, 0, 0, ALIGNED2, None) == -3      # odd ld
    assert rh(ALIGNED, 16, 16, 16, 0, 0, ALIGNED2 + 2, None) == -3  # out not 4-byte aligned
    assert qc(ALIGNED + 4, None) == -3                              # 64-bit counters need 8 bytes
    assert ph(ALIGNED + 4, 16, None) == -3
    sr = L.nvfp4_test_sr_round
    sr.restype = ctypes.c_int
    sr.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    assert sr(None, ALIGNED, 4, 6.0, ALIGNED2, None) == -1
    assert sr(ALIGNED, ALIGNED, -1, 6.0, ALIGNED2, None) == -2      # negative count
    assert sr(ALIGNED, ALIGNED, 4, 5.0, ALIGNED2, None) == -2       # Q other than 6 or 4
    assert sr(ALIGNED + 2, ALIGNED, 4, 4.0, ALIGNED2, None) == -3   # values not 4-byte aligned
    assert sr(ALIGNED, ALIGNED, 0, 6.0, ALIGNED2, None) == 0        # nothing to do, nothing launched
    gn = L.nvfp4_test_gemm_no_copy
    gn.restype = ctypes.c_int
    gn.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    gok = [ALIGNED, ALIGNED2, ALIGNED3, ALIGNED, ALIGNED2, ALIGNED3, ALIGNED, 128, 256, 256, 256, 1, ALIGNED3, None]
    gcall = lambda changes: gn(*[changes.get(i, v) for i, v in enumerate(gok)])
    assert gcall({0: None}) == -1 and gcall({12: None}) == -1        # operands, status required
    assert gcall({7: 100}) == -2 and gcall({9: 128}) == -2           # M % 128, K % 256
    assert gcall({10: 128}) == -2                                    # ldd < N
    assert gcall({0: ALIGNED + 8}) == -3 and gcall({10: 260}) == -3  # qa alignment, ldd % 8 with bf16
    nc = L.nvfp4_test_quantize_no_copy
    nc.restype = ctypes.c_int
    nc.argtypes = ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 7 +
                   [ctypes.c_int, ctypes.c_void_p])
    ok = [ALIGNED, 64, 256, 256, ALIGNED2, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED3, ALIGNED3, 0, None]
    call = lambda changes: nc(*[changes.get(i, v) for i, v in enumerate(ok)])
    assert call({0: None}) == -1 and call({10: None}) == -1         # x, status required
    assert call({1: 24}) == -2 and call({2: 24, 3: 24}) == -2       # M % 16, N % 16
    assert call({3: 128}) == -2                                     # ld < N
    assert call({0: ALIGNED + 8}) == -3 and call({5: ALIGNED + 4}) == -3
    assert call({11: 2}) == -4                                      # sr other than 0 or 1
