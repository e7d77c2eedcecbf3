"""GPU parity of the NVFP4 GEMM (nvfp4_gemm, tcgen05 block-scaled MMA) against
the oracle: both operands are quantized by the library with the tiled scale
layout (the MMA's operand format), the oracle multiplies the same codes and
scales (plain layout) after dequantizing them.

Tolerance.  Each product val_a * s_a * val_b * s_b is exact in the tensor
cores and the oracle's dequantized products differ from it by the rounding of
val * e4m3 * alpha to fp32 (2^-24 relative per operand); the tensor cores sum
the K products in fp32.  The bar is |D - D_ref| <= 2^-12 * sum_k |xa * xb| per
element (measured: at most 1e-6 on these shapes, fp32 accumulation), far
below the O(1) relative errors of a wrong scale, layout or operand order.  A
bf16 result is compared with the fp32 one rounded to bf16 (nearest even).
"""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_gb300 as nv
import oracle
import synthetic
from gpu_helpers import to_device

pytestmark = pytest.mark.gpu
ROW, COL, F46, SWZ = 1, 2, 64, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nv.build()
    oracle.build()


def operand(rows, K, seed, flags=ROW):
    """Quantize a (rows x K) tensor rowwise twice: tiled scales (for the GEMM)
    and plain scales (for the oracle); codes are identical."""
    bits = synthetic.activation_outlier_channels(rows, K, seed, frac=0.01)
    x = to_device(bits)
    amax = nv.nvfp4_amax(x, flags)
    tiled = nv.nvfp4_quantize(x, amax, flags | SWZ, 1)
    plain = nv.nvfp4_quantize(x, amax, flags, 1)
    torch.cuda.synchronize()
    assert torch.equal(tiled.q_row, plain.q_row)
    return tiled, plain


def check(M, N, K, seed=1, flags=ROW):
    A, Ap = operand(M, K, seed, flags)
    B, Bp = operand(N, K, seed + 100, flags)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = nv.nvfp4_gemm(A.q_row, A.s_row, A.alpha[0:1], B.q_row, B.s_row, B.alpha[0:1], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qa, sa, qb, sb = (t.cpu().numpy() for t in (Ap.q_row, Ap.s_row, Bp.q_row, Bp.s_row))
    aa, ab = float(Ap.alpha[0].item()), float(Bp.alpha[0].item())
    ref = oracle.gemm(qa, sa, aa, qb, sb, ab, K)
    xa = np.abs(oracle.dequantize(qa, sa, aa, M, K).astype(np.float64))
    xb = np.abs(oracle.dequantize(qb, sb, ab, N, K).astype(np.float64))
    mag = xa @ xb.T
    got = d.cpu().numpy()
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    rel = float((err / np.maximum(mag, 1e-30)).max())
    assert np.isfinite(got).all()
    assert rel <= 2.0 ** -16, f"max error {rel:.3e} of sum |xa*xb|"
    d16 = nv.nvfp4_gemm(A.q_row, A.s_row, A.alpha[0:1], B.q_row, B.s_row, B.alpha[0:1], out_dtype=torch.bfloat16,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(d16.view(torch.int16), d.to(torch.bfloat16).view(torch.int16))
    return rel


def test_gemm_single_tile_one_k_step():
    check(128, 128, 256)


@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (128, 256, 2048), (384, 128, 4096), (2048, 3072, 512),
                                   (2048, 2560, 768)])
def test_gemm_tiles_and_pipeline_stages(M, N, K):
    """Both tile widths (128 x 256 where N is a multiple of 256, else
    128 x 128), several output tiles per CTA (the last two shapes have more
    tiles than SMs: the accumulators are reused, and with three K steps per
    tile the four-stage ring wraps within a CTA's second tile), and K
    spanning more K steps than pipeline stages."""
    check(M, N, K, seed=M + N + K)


def test_gemm_with_four_over_six_operands():
    """4/6 picks per block between two scales; the MMA takes each block's byte."""
    check(256, 256, 1024, seed=7, flags=ROW | F46)


def test_gemm_rejects_bad_shapes_and_alignment():
    q = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((128, 16), dtype=torch.uint8, device="cuda")
    al = torch.ones(1, device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemm(q[:100], s, al, q, s, al)                    # M % 128
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemm(q[:, :64], s, al, q[:, :64], s, al)          # K = 128 < 256


@pytest.mark.parametrize("N", [256, 384])
def test_gemm_wait_timeout_is_reported_and_the_context_stays_usable(N):
    """The GEMM in a variant whose operand copies are never issued (test-only
    library; both tile widths): every bounded wait runs out, the kernel
    reports NVFP4_ERR_PIPELINE, drains and frees its tensor memory, and the
    next GEMM on the same context is correct."""
    import ctypes
    from gpu_helpers import selftest_lib
    hook = selftest_lib().nvfp4_test_gemm_no_copy
    hook.restype = ctypes.c_int
    hook.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    M, K = 256, 512
    A, _ = operand(M, K, 31)
    B, _ = operand(N, K, 32)
    d = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hook(A.q_row.data_ptr(), A.s_row.data_ptr(), A.alpha[0:1].data_ptr(), B.q_row.data_ptr(),
                B.s_row.data_ptr(), B.alpha[0:1].data_ptr(), d.data_ptr(), M, N, K, N, 0, status.data_ptr(),
                None) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == -8
    check(M, N, K, seed=33)  # the context is usable and the product kernel correct
