// quant1d.cu -- fused rowwise + columnwise NVFP4 quantization with 1x16 blocks.
//
// One read of X produces both copies: each thread loads a 16-row x 8-column
// register tile with sixteen coalesced 128-bit loads.  Rowwise blocks (16
// consecutive columns) span a lane pair and combine with one shuffle;
// columnwise blocks (16 consecutive rows of one column) lie entirely in one
// thread, so the transposed copy needs no shared-memory transpose.
//
// Sources: "Four Over Six (4/6)" technical summary (Problem statement,
// Methodology, Implementation details) and "Pretraining Large Language Models
// with NVFP4" sections 1, 2b and 2d.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

// Codes of 8 values of one block at scale s (block maximum Q): RN through the
// saturating cvt (clamped to +-4 first when a max-4 scale is subnormal and
// |v| could exceed 5), or SR with the given words.
template <bool SR>
__device__ __forceinline__ uint32_t quant8(const float* z, const BlockScale& s, float Q,
                                           const uint32_t* w) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(z[j], s.inv);
  if (SR) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = sr_round(v[j], Q, w[j]);
  } else if (Q == 4.0f && s.e < 8u) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fminf(fmaxf(v[j], -4.0f), 4.0f);
  }
  return e2m1x8(v);
}

__device__ __forceinline__ uint2 ctr_of(uint64_t i) { return make_uint2((uint32_t)i, (uint32_t)(i >> 32)); }

template <bool ROW, bool COL, bool Q46, bool SR>
__global__ void __launch_bounds__(kThreads) quant1d_kernel(const QuantArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool odd = (lane & 1) != 0;
  const int64_t r0 = ((int64_t)blockIdx.y * kWarps + warp) * 16;
  const int64_t c0 = (int64_t)blockIdx.x * kTileCols + lane * 8;

  // a2: alpha = amax / (6*448), or amax / (6*256) with 4/6
  const float den = Q46 ? kAlphaDen46 : kAlphaDen;
  const float A_r = a.amax[0], A_c = a.amax[1];
  const float alpha_r = __fdiv_rn(A_r, den);
  const float alpha_c = __fdiv_rn(A_c, den);
  const int st_r = ROW ? amax_status(A_r) : 0;
  const int st_c = COL ? amax_status(A_c) : 0;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha_r;
    a.alpha[1] = alpha_c;
    if ((st_r || st_c) && a.status) *a.status = st_r ? st_r : st_c;
  }
  if (st_r || st_c) return;
  if (r0 >= a.M) return;  // whole warp beyond the tensor

  const bool col_ok = c0 < a.N;
  const int sel = a.sel;

  // a3: one read of the 16x8 register tile
  uint32_t xr[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok && r0 + i < a.M) v = ld_stream(a.x + (r0 + i) * a.ld + c0);
    xr[i][0] = v.x;
    xr[i][1] = v.y;
    xr[i][2] = v.z;
    xr[i][3] = v.w;
  }
  const uint32_t signs = (a.rht_row || a.rht_col) ? rht_sign_bits(a.rht_k0, a.rht_k1) : 0u;
  const int64_t N = a.N, M = a.M;

  // Stochastic rounding without 4/6 and without a rowwise transform: one
  // Philox call per element feeds both copies (word 0 rowwise, word 1
  // columnwise) in a single sweep over column pairs.
  constexpr bool kFusedSR = SR && !Q46 && ROW && COL;
  if (kFusedSR && !a.rht_row) {
    float invR[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float b = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) b = fmaxf(b, fmaxf(fabsf(bf16_lo(xr[i][k])), fabsf(bf16_hi(xr[i][k]))));
      b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
      const BlockScale s = block_scale(b, alpha_r, 6.0f);
      invR[i] = s.inv;
      if (col_ok && !odd) a.s_row[(r0 + i) * (N / 16) + c0 / 16] = (uint8_t)s.e;
    }
    uint32_t rq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) rq[i] = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float z0[16], z1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        z0[i] = bf16_lo(xr[i][k]);
        z1[i] = bf16_hi(xr[i][k]);
      }
      if (a.rht_col) {
        rht16(z0, signs);
        rht16(z1, signs);
      }
      float b0 = 0.0f, b1 = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        b0 = fmaxf(b0, fabsf(z0[i]));
        b1 = fmaxf(b1, fabsf(z1[i]));
      }
      const BlockScale sc0 = block_scale(b0, alpha_c, 6.0f);
      const BlockScale sc1 = block_scale(b1, alpha_c, 6.0f);
      const int64_t ca = c0 + 2 * k, cb = ca + 1;
      uint32_t cqa[2] = {0u, 0u}, cqb[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint64_t base0 = a.ctr_off + (uint64_t)(r0 + i) * (uint64_t)N + (uint64_t)ca;
        const uint64_t base1 = base0 + (uint64_t)N;
        const uint2 c00 = ctr_of(base0), c01 = ctr_of(base0 + 1), c10 = ctr_of(base1), c11 = ctr_of(base1 + 1);
        const uint2 w00 = philox_w01(c00.x, c00.y, a.sr_k0, a.sr_k1);  // (i,   ca)
        const uint2 w01 = philox_w01(c01.x, c01.y, a.sr_k0, a.sr_k1);  // (i,   cb)
        const uint2 w10 = philox_w01(c10.x, c10.y, a.sr_k0, a.sr_k1);  // (i+1, ca)
        const uint2 w11 = philox_w01(c11.x, c11.y, a.sr_k0, a.sr_k1);  // (i+1, cb)
        // rowwise codes (word 0), values are the untransformed x
        const float r00 = sr_round(__fmul_rn(bf16_lo(xr[i][k]), invR[i]), 6.0f, w00.x);
        const float r01 = sr_round(__fmul_rn(bf16_hi(xr[i][k]), invR[i]), 6.0f, w01.x);
        const float r10 = sr_round(__fmul_rn(bf16_lo(xr[i + 1][k]), invR[i + 1]), 6.0f, w10.x);
        const float r11 = sr_round(__fmul_rn(bf16_hi(xr[i + 1][k]), invR[i + 1]), 6.0f, w11.x);
        rq[i] |= e2m1x2(r00, r01) << (8 * k);
        rq[i + 1] |= e2m1x2(r10, r11) << (8 * k);
        // columnwise codes (word 1)
        const float g0a = sr_round(__fmul_rn(z0[i], sc0.inv), 6.0f, w00.y);
        const float g1a = sr_round(__fmul_rn(z0[i + 1], sc0.inv), 6.0f, w10.y);
        const float g0b = sr_round(__fmul_rn(z1[i], sc1.inv), 6.0f, w01.y);
        const float g1b = sr_round(__fmul_rn(z1[i + 1], sc1.inv), 6.0f, w11.y);
        cqa[i / 8] |= e2m1x2(g0a, g1a) << (8 * ((i / 2) % 4));
        cqb[i / 8] |= e2m1x2(g0b, g1b) << (8 * ((i / 2) % 4));
      }
      if (col_ok) {
        *reinterpret_cast<uint2*>(a.q_col + ca * (M / 2) + r0 / 2) = make_uint2(cqa[0], cqa[1]);
        *reinterpret_cast<uint2*>(a.q_col + cb * (M / 2) + r0 / 2) = make_uint2(cqb[0], cqb[1]);
        a.s_col[ca * (M / 16) + r0 / 16] = (uint8_t)sc0.e;
        a.s_col[cb * (M / 16) + r0 / 16] = (uint8_t)sc1.e;
      }
    }
    if (col_ok) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<uint32_t*>(a.q_row + (r0 + i) * (N / 2) + c0 / 2) = rq[i];
    }
    return;
  }

  // ---- rowwise copy: blocks of 16 columns, split over a lane pair
  if (ROW) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = r0 + i;
      if (r >= M) break;  // same row for every lane of the warp
      float z[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        z[2 * k] = bf16_lo(xr[i][k]);
        z[2 * k + 1] = bf16_hi(xr[i][k]);
      }
      if (a.rht_row) rht16_pair(z, signs, odd);
      float b = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) b = fmaxf(b, fabsf(z[j]));
      b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
      uint32_t w[8];
      if (SR) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint2 c = ctr_of(a.ctr_off + (uint64_t)r * (uint64_t)N + (uint64_t)(c0 + j));
          w[j] = philox_w01(c.x, c.y, a.sr_k0, a.sr_k1).x;
        }
      }
      const BlockScale s6 = block_scale(b, alpha_r, 6.0f);
      uint32_t codes = quant8<SR>(z, s6, 6.0f, w);
      uint32_t e = s6.e;
      if (Q46) {
        const BlockScale s4 = block_scale(b, alpha_r, 4.0f);
        const uint32_t codes4 = quant8<SR>(z, s4, 4.0f, w);
        float sc6 = score8(z, codes, s6.d, sel);
        float sc4 = score8(z, codes4, s4.d, sel);
        sc6 = err_combine(sc6, __shfl_xor_sync(0xFFFFFFFFu, sc6, 1), sel);
        sc4 = err_combine(sc4, __shfl_xor_sync(0xFFFFFFFFu, sc4, 1), sel);
        if (sc4 < sc6) {
          codes = codes4;
          e = s4.e;
        }
      }
      if (col_ok) {
        *reinterpret_cast<uint32_t*>(a.q_row + r * (N / 2) + c0 / 2) = codes;
        if (!odd) a.s_row[r * (N / 16) + c0 / 16] = (uint8_t)e;
      }
    }
  }

  // ---- columnwise copy: blocks of 16 rows of one column, all in this thread
  if (COL) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int k = cc >> 1;
      float z[16];
      if (cc & 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = bf16_hi(xr[i][k]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = bf16_lo(xr[i][k]);
      }
      const int64_t c = c0 + cc;
      if (a.rht_col) rht16(z, signs);
      float b = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(z[i]));
      uint32_t w[16];
      if (SR) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint2 ct = ctr_of(a.ctr_off + (uint64_t)(r0 + i) * (uint64_t)N + (uint64_t)c);
          w[i] = philox_w01(ct.x, ct.y, a.sr_k0, a.sr_k1).y;
        }
      }
      const BlockScale s6 = block_scale(b, alpha_c, 6.0f);
      uint32_t lo = quant8<SR>(z, s6, 6.0f, w);
      uint32_t hi = quant8<SR>(z + 8, s6, 6.0f, w + 8);
      uint32_t e = s6.e;
      if (Q46) {
        const BlockScale s4 = block_scale(b, alpha_c, 4.0f);
        const uint32_t lo4 = quant8<SR>(z, s4, 4.0f, w);
        const uint32_t hi4 = quant8<SR>(z + 8, s4, 4.0f, w + 8);
        const float sc6 = err_combine(score8(z, lo, s6.d, sel), score8(z + 8, hi, s6.d, sel), sel);
        const float sc4 = err_combine(score8(z, lo4, s4.d, sel), score8(z + 8, hi4, s4.d, sel), sel);
        if (sc4 < sc6) {
          lo = lo4;
          hi = hi4;
          e = s4.e;
        }
      }
      if (col_ok) {
        *reinterpret_cast<uint2*>(a.q_col + c * (M / 2) + r0 / 2) = make_uint2(lo, hi);
        a.s_col[c * (M / 16) + r0 / 16] = (uint8_t)e;
      }
    }
  }
}

template <bool ROW, bool COL, bool Q46, bool SR>
cudaError_t launch(const QuantArgs& a, cudaStream_t s) {
  quant1d_kernel<ROW, COL, Q46, SR><<<tile_grid(a.M, a.N), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <bool ROW, bool COL>
cudaError_t launch_rc(const QuantArgs& a, bool q46, bool sr, cudaStream_t s) {
  if (q46) return sr ? launch<ROW, COL, true, true>(a, s) : launch<ROW, COL, true, false>(a, s);
  return sr ? launch<ROW, COL, false, true>(a, s) : launch<ROW, COL, false, false>(a, s);
}

}  // namespace

cudaError_t launch_quant1d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t s) {
  if (row && col) return launch_rc<true, true>(a, q46, sr, s);
  if (row) return launch_rc<true, false>(a, q46, sr, s);
  return launch_rc<false, true>(a, q46, sr, s);
}

}  // namespace nvfp4
