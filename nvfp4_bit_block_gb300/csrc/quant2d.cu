// quant2d.cu -- NVFP4 quantization with 16x16 2D block scales (weights).
//
// "Pretraining Large Language Models with NVFP4" section 2c: one scale per
// 16x16 tile shared by the forward (rowwise) and the transposed (columnwise)
// copy, so both copies hold the same quantized weight.  A lane pair holds one
// tile (16 rows x 8 columns each); every element is quantized once and its
// code is packed into both layouts, so C's codes are exactly the transpose of
// R's.  With 4/6 the tile is scored at block maximum 6 and 4 over all 256
// elements ("Four Over Six (4/6)" technical summary, Methodology).
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

__device__ __forceinline__ uint32_t word0_of(const QuantArgs& a, int64_t r, int64_t c) {
  const uint64_t i = a.ctr_off + (uint64_t)r * (uint64_t)a.N + (uint64_t)c;
  return philox_w01((uint32_t)i, (uint32_t)(i >> 32), a.sr_k0, a.sr_k1).x;
}

// Scaled (and, for SR, rounded) value of one element at block scale s.
template <bool SR>
__device__ __forceinline__ float scaled(float z, const BlockScale& s, float Q, uint32_t w) {
  float v = __fmul_rn(z, s.inv);
  if (SR) return sr_round(v, Q, w);
  if (Q == 4.0f && s.e < 8u) v = fminf(fmaxf(v, -4.0f), 4.0f);
  return v;
}

// 4/6 score of the whole 16x16 tile at scale s: per row a tree over this
// lane's 8 columns, plus the partner's half, then a tree over the 16 rows.
template <bool SR>
__device__ __forceinline__ float tile_score(const uint32_t (&xr)[16][4], const BlockScale& s, float Q,
                                            const QuantArgs& a, int64_t r0, int64_t c0, int sel) {
  float rows[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float z[8], v[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      z[2 * k] = bf16_lo(xr[i][k]);
      z[2 * k + 1] = bf16_hi(xr[i][k]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = scaled<SR>(z[j], s, Q, SR ? word0_of(a, r0 + i, c0 + j) : 0u);
    const float part = score8(z, e2m1x8(v), s.d, sel);
    rows[i] = err_combine(part, __shfl_xor_sync(0xFFFFFFFFu, part, 1), sel);
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i += 2 * h) rows[i] = err_combine(rows[i], rows[i + h], sel);
  }
  return rows[0];
}

template <bool ROW, bool COL, bool Q46, bool SR>
__global__ void __launch_bounds__(kThreads) quant2d_kernel(const QuantArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool odd = (lane & 1) != 0;
  const int64_t r0 = ((int64_t)blockIdx.y * kWarps + warp) * 16;
  const int64_t c0 = (int64_t)blockIdx.x * kTileCols + lane * 8;

  const float den = Q46 ? kAlphaDen46 : kAlphaDen;
  const float A = a.amax[0];
  const float alpha = __fdiv_rn(A, den);
  const int st = amax_status(A);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha;
    a.alpha[1] = __fdiv_rn(a.amax[1], den);
    if (st && a.status) *a.status = st;
  }
  if (st) return;
  if (r0 >= a.M) return;

  const bool col_ok = c0 < a.N;
  const int64_t N = a.N, M = a.M;
  uint32_t xr[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok) v = ld_stream(a.x + (r0 + i) * a.ld + c0);
    xr[i][0] = v.x;
    xr[i][1] = v.y;
    xr[i][2] = v.z;
    xr[i][3] = v.w;
  }

  // a5: tile maximum over 256 values (this lane's 128, then the partner's)
  float b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) b = fmaxf(b, fmaxf(fabsf(bf16_lo(xr[i][k])), fabsf(bf16_hi(xr[i][k]))));
  b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));

  BlockScale s = block_scale(b, alpha, 6.0f);
  float Q = 6.0f;
  if (Q46) {
    const BlockScale s4 = block_scale(b, alpha, 4.0f);
    const float sc6 = tile_score<SR>(xr, s, 6.0f, a, r0, c0, a.sel);
    const float sc4 = tile_score<SR>(xr, s4, 4.0f, a, r0, c0, a.sel);
    if (sc4 < sc6) {
      s = s4;
      Q = 4.0f;
    }
  }

  // a7 + a9: each element once, packed rowwise (pairs along a row) and
  // columnwise (pairs along a column)
  uint32_t cq[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) cq[j][0] = cq[j][1] = 0u;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float v0[8], v1[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v0[2 * k] = scaled<SR>(bf16_lo(xr[i][k]), s, Q, SR ? word0_of(a, r0 + i, c0 + 2 * k) : 0u);
      v0[2 * k + 1] = scaled<SR>(bf16_hi(xr[i][k]), s, Q, SR ? word0_of(a, r0 + i, c0 + 2 * k + 1) : 0u);
      v1[2 * k] = scaled<SR>(bf16_lo(xr[i + 1][k]), s, Q, SR ? word0_of(a, r0 + i + 1, c0 + 2 * k) : 0u);
      v1[2 * k + 1] =
          scaled<SR>(bf16_hi(xr[i + 1][k]), s, Q, SR ? word0_of(a, r0 + i + 1, c0 + 2 * k + 1) : 0u);
    }
    if (ROW && col_ok) {
      *reinterpret_cast<uint32_t*>(a.q_row + (r0 + i) * (N / 2) + c0 / 2) = e2m1x8(v0);
      *reinterpret_cast<uint32_t*>(a.q_row + (r0 + i + 1) * (N / 2) + c0 / 2) = e2m1x8(v1);
    }
    if (COL) {
#pragma unroll
      for (int j = 0; j < 8; ++j) cq[j][i / 8] |= e2m1x2(v0[j], v1[j]) << (8 * ((i / 2) % 4));
    }
  }
  if (!col_ok) return;
  if (COL) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      *reinterpret_cast<uint2*>(a.q_col + (c0 + j) * (M / 2) + r0 / 2) = make_uint2(cq[j][0], cq[j][1]);
      a.s_col[(c0 + j) * (M / 16) + r0 / 16] = (uint8_t)s.e;
    }
  }
  if (ROW && !odd) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a.s_row[(r0 + i) * (N / 16) + c0 / 16] = (uint8_t)s.e;
  }
}

template <bool ROW, bool COL, bool Q46, bool SR>
cudaError_t launch(const QuantArgs& a, cudaStream_t st) {
  quant2d_kernel<ROW, COL, Q46, SR><<<tile_grid(a.M, a.N), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <bool ROW, bool COL>
cudaError_t launch_rc(const QuantArgs& a, bool q46, bool sr, cudaStream_t st) {
  if (q46) return sr ? launch<ROW, COL, true, true>(a, st) : launch<ROW, COL, true, false>(a, st);
  return sr ? launch<ROW, COL, false, true>(a, st) : launch<ROW, COL, false, false>(a, st);
}

}  // namespace

cudaError_t launch_quant2d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t st) {
  if (row && col) return launch_rc<true, true>(a, q46, sr, st);
  if (row) return launch_rc<true, false>(a, q46, sr, st);
  return launch_rc<false, true>(a, q46, sr, st);
}

}  // namespace nvfp4
