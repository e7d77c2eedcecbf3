#pragma once
// quant1d_kernel.cuh -- NVFP4 quantization with 1x16 blocks: the rowwise copy
// and/or the columnwise (transposed) copy from one read of X.
//
// Tiles.  Persistent CTAs stream 64 x 256 bf16 tiles into two shared-memory
// buffers with TMA bulk tensor copies (four 64 x 64 boxes, 128-byte swizzle,
// completion on an mbarrier with a bounded wait); one thread issues the next
// tile's copies while the CTA works on the current one.
//
// Threads.  Four threads share each 16 x 16 sub-tile, one 8 x 8 patch each:
// lane bit 0 picks the column half, lane bit 4 the row half, lane bits 1-3
// the sub-tile along the row, so a warp covers 16 rows x 128 columns and the
// CTA's eight warps cover the tile.  A rowwise block (16 values of a row) is
// split between lanes l and l^1, a columnwise block (16 values of a column)
// between lanes l and l^16; block maxima, 4/6 scores and the last Hadamard
// stage are combined with one shuffle, in the same order of operations as a
// single thread holding the block would use.  A thread reads its patch once
// (eight 16-byte shared loads, conflict-free under the swizzle) and keeps it
// as bf16 pairs in registers.
//   - rowwise: patch row by patch row; a half row's eight codes are one
//     32-bit word, stored directly (a quarter warp writes 32 contiguous bytes);
//   - columnwise: patch column pair by column pair (one bf16x2 word per patch
//     row); a half column's eight codes are one word, staged in shared memory
//     and written as 32 bytes per column of the transposed copy.
// With stochastic rounding on both copies (without 4/6 and without a rowwise
// Hadamard transform) a single pass in column-pair order serves both copies
// from one Philox4x32-10 call per element (word 0 rowwise, word 1
// columnwise), the rowwise words assembled byte by byte.  The other
// stochastic-rounding combinations draw each copy's word in its own pass.
//
// Per block the scale byte comes from a division-free quotient (see
// quotient_rn) and (d, 1/d) from a per-CTA table of the 127 scale values; the
// RHT flags, the 4/6 rule and the rounding mode are template parameters, so
// the block code is straight-line.
//
// Sources: "Four Over Six (4/6)" technical summary (Problem statement,
// Methodology, Implementation details) and "Pretraining Large Language Models
// with NVFP4" sections 1, 2b and 2d.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tile_pipeline.cuh"
#include "tma.cuh"

namespace nvfp4 {
namespace q1d {

using tile::kTM;
using tile::kTN;
constexpr int kBlockThreads = 256;
constexpr uint32_t kFull = 0xFFFFFFFFu;
// two tile buffers, the column staging (codes, scales) and the two (d, 1/d)
// tables: 76,800 bytes, so that three CTAs fit in an SM
constexpr int kSmemBytes = 2 * tile::kTileBytes + tile::kCStageBytes + tile::kSStageBytes + 256 * 8;

// Staging position of tile column c: columns 16 apart are XOR-shifted within
// their group of 8 so that the 16 lanes of a half warp, which hold columns
// 8 apart, write to 16 different banks.  A permutation of 0..255.
__device__ __forceinline__ int stage_col(int c) { return c ^ ((c >> 4) & 7); }

// Per-copy scale constants: den = Q*alpha and its correctly rounded
// reciprocal for Q = 6 and Q = 4, and the copy's (d, 1/d) table.
struct CopyScales {
  float den6, rden6, den4, rden4;
  const float2* tbl;
};

__device__ __forceinline__ CopyScales make_scales(float alpha, const float2* tbl) {
  CopyScales c;
  c.den6 = __fmul_rn(6.0f, alpha);
  c.den4 = __fmul_rn(4.0f, alpha);
  c.rden6 = (c.den6 != 0.0f) ? __frcp_rn(c.den6) : 0.0f;
  c.rden4 = (c.den4 != 0.0f) ? __frcp_rn(c.den4) : 0.0f;
  c.tbl = tbl;
  return c;
}

// Scale bytes of a block with maximum b (e4 only with 4/6).
template <bool Q46>
__device__ __forceinline__ void block_bytes(float b, const CopyScales& sc, uint32_t& e6, uint32_t& e4) {
  e6 = scale_byte(b, sc.den6, sc.rden6);
  e4 = Q46 ? scale_byte(b, sc.den4, sc.rden4) : 0u;
}

// Philox words 0 and 1 of source element index i (64-bit, modulo 2^64).
__device__ __forceinline__ uint2 words_of(uint64_t i, uint32_t k0, uint32_t k1) {
  return philox_w01((uint32_t)i, (uint32_t)(i >> 32), k0, k1);
}

// Scaled values of a candidate: v = z * (1/d), then stochastic rounding, or
// for a max-4 candidate whose scale byte is subnormal or saturated the clamp
// to +-4 that round-to-nearest needs.
template <bool SR>
__device__ __forceinline__ void scale8(const float* z, float inv, uint32_t e, float Q, const uint32_t* w, float* v) {
  const float2 inv2 = make_float2(inv, inv);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 r = mul2(make_float2(z[2 * j], z[2 * j + 1]), inv2);
    v[2 * j] = r.x;
    v[2 * j + 1] = r.y;
  }
  if (SR) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = sr_round(v[j], Q, w[j]);
  } else if (Q == 4.0f && max4_needs_clamp(e)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fminf(fmaxf(v[j], -4.0f), 4.0f);
  }
}

// Error terms of a pair: err = z - val*d rounded once, then |err| (MAE,
// MAXERR) or err*err (MSE); the pair's first tree level.
template <int SEL>
__device__ __forceinline__ float pair_term(float e0, float e1) {
  if (SEL == kSelMSE) return __fadd_rn(__fmul_rn(e0, e0), __fmul_rn(e1, e1));
  if (SEL == kSelMax) return fmaxf(fabsf(e0), fabsf(e1));
  return __fadd_rn(fabsf(e0), fabsf(e1));
}

// One 4/6 candidate on a half row (8 values in block order): its code word
// and the score of the half, a perfect binary tree over the 8 terms.
template <bool SR, int SEL>
__device__ __forceinline__ float cand8(const float* z, uint32_t e, float2 di, float Q, const uint32_t* w,
                                       uint32_t& codes) {
  float v[8];
  scale8<SR>(z, di.y, e, Q, w, v);
  uint32_t h[4];
  codes = e2m1x8_enc_dec(v, h);
  const float2 nd = make_float2(-di.x, -di.x);
  float t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 err = fma2(f16x2_to_f32x2(h[k]), nd, make_float2(z[2 * k], z[2 * k + 1]));
    t[k] = pair_term<SEL>(err.x, err.y);
  }
  return err_combine(err_combine(t[0], t[1], SEL), err_combine(t[2], t[3], SEL), SEL);
}

// Both columns of a column pair: zp[i] = (column a, column b) at patch row i.
// Scaled values per row as packed pairs; codes of rows 2m, 2m+1 of a column
// are byte m of that column's word.
template <bool SR>
__device__ __forceinline__ void scale8x2(const float2* zp, float inva, float invb, uint32_t ea, uint32_t eb, float Q,
                                         const uint32_t* wa, const uint32_t* wb, float2* v) {
  const float2 inv2 = make_float2(inva, invb);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = mul2(zp[i], inv2);
  if (SR) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i].x = sr_round(v[i].x, Q, wa[i]);
      v[i].y = sr_round(v[i].y, Q, wb[i]);
    }
  } else if (Q == 4.0f) {
    if (max4_needs_clamp(ea)) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i].x = fminf(fmaxf(v[i].x, -4.0f), 4.0f);
    }
    if (max4_needs_clamp(eb)) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i].y = fminf(fmaxf(v[i].y, -4.0f), 4.0f);
    }
  }
}

// Code words of both columns of a pair (no 4/6).
__device__ __forceinline__ uint2 encode8x2(const float2* v) {
  uint32_t ba[4], bb[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    ba[m] = e2m1x2(v[2 * m].x, v[2 * m + 1].x);
    bb[m] = e2m1x2(v[2 * m].y, v[2 * m + 1].y);
  }
  return make_uint2(pack4(ba[0], ba[1], ba[2], ba[3]), pack4(bb[0], bb[1], bb[2], bb[3]));
}

// One 4/6 candidate on both half columns of a pair: code words and the two
// half scores (tree over rows 0..7 of each column).
template <bool SR, int SEL>
__device__ __forceinline__ float2 cand8x2(const float2* zp, uint32_t ea, uint32_t eb, float2 dia, float2 dib, float Q,
                                          const uint32_t* wa, const uint32_t* wb, uint2& codes) {
  float2 v[8];
  scale8x2<SR>(zp, dia.y, dib.y, ea, eb, Q, wa, wb, v);
  uint32_t ba[4], bb[4];
  float ta[4], tb[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t ha, hb;
    ba[m] = e2m1x2_enc_dec(v[2 * m].x, v[2 * m + 1].x, ha);
    bb[m] = e2m1x2_enc_dec(v[2 * m].y, v[2 * m + 1].y, hb);
    const float2 va = f16x2_to_f32x2(ha), vb = f16x2_to_f32x2(hb);
    ta[m] = pair_term<SEL>(__fmaf_rn(-va.x, dia.x, zp[2 * m].x), __fmaf_rn(-va.y, dia.x, zp[2 * m + 1].x));
    tb[m] = pair_term<SEL>(__fmaf_rn(-vb.x, dib.x, zp[2 * m].y), __fmaf_rn(-vb.y, dib.x, zp[2 * m + 1].y));
  }
  codes = make_uint2(pack4(ba[0], ba[1], ba[2], ba[3]), pack4(bb[0], bb[1], bb[2], bb[3]));
  if (SEL == kSelMax)
    return make_float2(fmaxf(fmaxf(ta[0], ta[1]), fmaxf(ta[2], ta[3])), fmaxf(fmaxf(tb[0], tb[1]), fmaxf(tb[2], tb[3])));
  const float2 s01 = add2(make_float2(ta[0], tb[0]), make_float2(ta[1], tb[1]));
  const float2 s23 = add2(make_float2(ta[2], tb[2]), make_float2(ta[3], tb[3]));
  return add2(s01, s23);
}

// Hadamard stages 1, 2, 4 of a half row (8 values, block positions
// 8*half + j): the full butterfly's first three stages only pair values inside
// aligned groups of 8.  Same operations as wht16.
__device__ __forceinline__ void wht8(float* z) {
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float a = z[i], b = z[i + 1];
    z[i] = __fadd_rn(a, b);
    z[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      if ((i & h) == 0) {
        const float2 a = make_float2(z[i], z[i + 1]), b = make_float2(z[i + h], z[i + h + 1]);
        const float2 s = add2(a, b), d = sub2(a, b);
        z[i] = s.x;
        z[i + 1] = s.y;
        z[i + h] = d.x;
        z[i + h + 1] = d.y;
      }
    }
  }
}

// The same three stages on a pair of half columns held as row pairs.
__device__ __forceinline__ void wht8_x2(float2* z) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float2 a = z[i], b = z[i + h];
        z[i] = add2(a, b);
        z[i + h] = sub2(a, b);
      }
    }
  }
}

// Last stage (pairs i, i + 8) across the two threads of a block: the thread
// with the first half keeps a + b, the other a - b, where a is the first
// half's value; then the 1/4 (exact).
__device__ __forceinline__ float2 last_stage(float2 mine, float2 theirs, bool second) {
  const float2 y = second ? sub2(theirs, mine) : add2(mine, theirs);
  return mul2(y, make_float2(0.25f, 0.25f));
}

// Write the staged columnwise outputs of one tile: tile column `c` (one per
// thread) gets its codes for up to 64 rows (32 bytes, four row blocks of 8)
// and up to 4 scales.  With swz the scales go to the tiled layout (their four
// row blocks stay four consecutive bytes there, as the tile origin is a
// multiple of 64 rows).
__device__ __forceinline__ void write_col_outputs(const uint8_t* cstage, const uint8_t* sstage, uint8_t* q_col,
                                                  uint8_t* s_col, int64_t M, int64_t N, tile::Coord tc, int c,
                                                  bool swz) {
  const int64_t gc = tc.C0 + c;
  if (gc >= N) return;
  int64_t nrb = (M - tc.R0) / 16;
  if (nrb > 4) nrb = 4;
  const int sc = stage_col(c);
  uint2 w[4];
#pragma unroll
  for (int rb = 0; rb < 4; ++rb) w[rb] = *reinterpret_cast<const uint2*>(cstage + rb * 2048 + sc * 8);
  uint8_t* dst = q_col + gc * (M / 2) + tc.R0 / 2;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(dst);
  if (nrb == 4 && (addr & 31) == 0) {
    tile::st_v8(dst, w[0], w[1], w[2], w[3]);
  } else if (nrb == 4 && (addr & 15) == 0) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0].x, w[0].y, w[1].x, w[1].y);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[2].x, w[2].y, w[3].x, w[3].y);
  } else {
    for (int rb = 0; rb < nrb; ++rb) *reinterpret_cast<uint2*>(dst + 8 * rb) = w[rb];
  }
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(sstage + sc * 4);
  uint8_t* sdst = s_col + (swz ? tile::sf_swz_off(gc, tc.R0 / 16, (M / 16 + 3) / 4) : gc * (M / 16) + tc.R0 / 16);
  if (nrb == 4 && (reinterpret_cast<uintptr_t>(sdst) & 3) == 0) {
    *reinterpret_cast<uint32_t*>(sdst) = sw;
  } else {
    for (int rb = 0; rb < nrb; ++rb) sdst[rb] = (uint8_t)(sw >> (8 * rb));
  }
}

// RHT bit 0: Hadamard on the rowwise copy; bit 1: on the columnwise copy.
// NOCOPY (a test instantiation only): arm the tile barriers but issue no copy.
template <bool ROW, bool COL, bool Q46, bool SR, int SEL, int RHT, bool NOCOPY = false>
__global__ void __launch_bounds__(kBlockThreads, SR ? 2 : 3)
    quant1d_kernel(const QuantArgs a, const __grid_constant__ CUtensorMap xmap) {
  constexpr bool kRhtRow = (RHT & 1) != 0, kRhtCol = (RHT & 2) != 0;
  // one pass in column-pair order serves both copies from one Philox call
  constexpr bool kOnePass = SR && ROW && COL && !Q46 && !kRhtRow;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bufs = smem;                                      // 2 x 32 KB tiles (1024-aligned)
  uint8_t* cstage = smem + 2 * tile::kTileBytes;             // 8 KB: [4 row blocks][256 columns] x 8 bytes
  uint8_t* sstage = cstage + tile::kCStageBytes;             // 1 KB: [256 columns] x 4 scale bytes
  float2* tbl = reinterpret_cast<float2*>(sstage + tile::kSStageBytes);  // 2 x 128 (d, 1/d)
  // Scale bytes never exceed 0x7E (448), so entry 127 of each table is free:
  // it holds the tile barrier of buffer 0 (R table) and buffer 1 (C table).
  const uint32_t bar0 = tile::smem_u32(tbl + 127), bar1 = tile::smem_u32(tbl + 255);

  // a2: alpha = amax / (6*448), or amax / (6*256) with 4/6
  const float den = Q46 ? kAlphaDen46 : kAlphaDen;
  const float A_r = a.amax[0], A_c = a.amax[1];
  const float alpha_r = __fdiv_rn(A_r, den);
  const float alpha_c = __fdiv_rn(A_c, den);
  const int st_r = ROW ? amax_status(A_r) : 0;
  const int st_c = COL ? amax_status(A_c) : 0;
  const bool misaligned = (tile::smem_u32(smem) & 1023u) != 0u;  // the 128-byte swizzle needs 1 KB alignment
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha_r;
    a.alpha[1] = alpha_c;
    if ((st_r || st_c) && a.status) *a.status = st_r ? st_r : st_c;
    if (misaligned && !(st_r || st_c) && a.status) *a.status = kStatusPipeline;
  }
  if (st_r || st_c || misaligned) return;

  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x;
  if ((tid & 127) != 127) tbl[tid] = scale_entry(tid & 127, (tid >> 7) ? alpha_c : alpha_r);
  if (tid == 0) {
    tma::mbar_init(bar0, 1);
    tma::mbar_init(bar1, 1);
    tma::fence_barrier_init();
  }
  __syncthreads();  // barriers and tables ready
  const CopyScales scR = make_scales(alpha_r, tbl);
  const CopyScales scC = make_scales(alpha_c, tbl + 128);
  const uint32_t signs = (kRhtRow || kRhtCol) ? rht_sign_bits(a.rht_k0, a.rht_k1) : 0u;

  // thread geometry (see the header comment)
  const int lane = tid & 31, warp = tid >> 5;
  const int ch = lane & 1, bcol = (lane >> 1) & 7, rh = lane >> 4;
  const int rb = warp >> 1;                                 // 16-row band of this warp
  const int tcol0 = 128 * (warp & 1) + 16 * bcol + 8 * ch;  // first tile column of the patch
  const int trow0 = 16 * rb + 8 * rh;                       // first tile row of the patch
  const int pc = (tcol0 & 63) >> 3;                         // the patch's 16-byte chunk within its box
  const uint32_t poff = (tcol0 >> 6) * 8192 + trow0 * 128;  // the patch's box and first row
  const int64_t hN = N / 2, sN = N / 16;

  auto issue = [&](int b, const tile::Coord& c) {
    const uint32_t bar = b ? bar1 : bar0;
    tma::arrive_expect_tx(bar, tile::kTileBytes);
    if (NOCOPY) return;
    const uint32_t dst = tile::smem_u32(bufs + b * tile::kTileBytes);
#pragma unroll
    for (int j = 0; j < 4; ++j) tma::load_2d(dst + j * 8192, &xmap, (int)c.C0 + 64 * j, (int)c.R0, bar);
  };

  tile::Walker w;
  w.init(M, N);
  if (tid == 0 && w.valid()) issue(0, w.coord());
  for (int it = 0; w.valid(); w = w.next(), ++it) {
    const int b = it & 1;
    const uint8_t* buf = bufs + b * tile::kTileBytes;
    if (tid == 0) {
      const tile::Walker wn = w.next();
      if (wn.valid()) issue(b ^ 1, wn.coord());  // that buffer was released by the last barrier
    }
    const uint32_t parity = (it >> 1) & 1;
    const bool arrived = tma::wait(b ? bar1 : bar0, parity);
    if (!__syncthreads_and(arrived)) {
      // a copy did not arrive in time: report it, give the copies in flight
      // one more bounded wait, and stop
      if (tid == 0) {
        if (a.status) atomicExch(a.status, kStatusPipeline);
        tma::wait(b ? bar1 : bar0, parity);
        if (w.next().valid()) tma::wait(b ? bar0 : bar1, ((it + 1) >> 1) & 1);
      }
      return;
    }
    const tile::Coord tc = w.coord();
    const int64_t grow0 = tc.R0 + trow0, gcol0 = tc.C0 + tcol0;
    // the sub-tile's 16 columns lie inside the tensor or outside it (N % 16 == 0)
    const bool cols_in = tc.C0 + (tcol0 & ~15) < N;

    const uint8_t* pbase = buf + poff;

    if (kOnePass) {
      // a3: the whole patch, eight rows of four bf16 pairs
      uint32_t wd[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 q = *reinterpret_cast<const uint4*>(pbase + i * 128 + ((pc ^ i) << 4));
        wd[i][0] = q.x;
        wd[i][1] = q.y;
        wd[i][2] = q.z;
        wd[i][3] = q.w;
      }
      // ---- both copies with stochastic rounding, one Philox call per element
      // rowwise scales of the 8 patch rows
      float inv_r[8];
      uint32_t e_r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t m = absmax_bf16x2(absmax_bf16x2(wd[i][0], wd[i][1]), absmax_bf16x2(wd[i][2], wd[i][3]));
        m = absmax_bf16x2(m, __shfl_xor_sync(kFull, m, 1)) & 0x7FFF7FFFu;
        uint32_t e4;
        block_bytes<false>(fmaxf(bf16_lo(m), bf16_hi(m)), scR, e_r[i], e4);
        inv_r[i] = scR.tbl[e_r[i]].y;
      }
      uint32_t rword[8];
      const uint64_t ctr0 = a.ctr_off + (uint64_t)grow0 * (uint64_t)N + (uint64_t)gcol0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 zp[8];
        float ba, bb;
        if (kRhtCol) {
#pragma unroll
          for (int i = 0; i < 8; ++i) zp[i] = bf16x2_to_f32x2(wd[i][k] ^ rht_mask_col(signs, 8 * rh + i));
          wht8_x2(zp);
          ba = 0.0f;
          bb = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 th = make_float2(__shfl_xor_sync(kFull, zp[i].x, 16), __shfl_xor_sync(kFull, zp[i].y, 16));
            zp[i] = last_stage(zp[i], th, rh != 0);
            ba = fmaxf(ba, fabsf(zp[i].x));
            bb = fmaxf(bb, fabsf(zp[i].y));
          }
          ba = fmaxf(ba, __shfl_xor_sync(kFull, ba, 16));
          bb = fmaxf(bb, __shfl_xor_sync(kFull, bb, 16));
        } else {
          uint32_t m = 0u;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            zp[i] = bf16x2_to_f32x2(wd[i][k]);
            m = absmax_bf16x2(m, wd[i][k]);
          }
          m = absmax_bf16x2(m, __shfl_xor_sync(kFull, m, 16)) & 0x7FFF7FFFu;
          ba = bf16_lo(m);
          bb = bf16_hi(m);
        }
        uint32_t ea, eb, e4;
        block_bytes<false>(ba, scC, ea, e4);
        block_bytes<false>(bb, scC, eb, e4);
        const float inva = scC.tbl[ea].y, invb = scC.tbl[eb].y;
        uint32_t ca[4], cb[4];
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
          float cv[2][2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = 2 * m2 + h;
            const uint64_t ci = ctr0 + (uint64_t)i * (uint64_t)N + (uint64_t)(2 * k);
            const uint2 wa = words_of(ci, a.sr_k0, a.sr_k1);
            const uint2 wb = words_of(ci + 1u, a.sr_k0, a.sr_k1);
            const float2 zr = kRhtCol ? bf16x2_to_f32x2(wd[i][k]) : zp[i];
            const float2 vr = mul2(zr, make_float2(inv_r[i], inv_r[i]));
            const uint32_t rbyte = e2m1x2(sr_round(vr.x, 6.0f, wa.x), sr_round(vr.y, 6.0f, wb.x));
            rword[i] = (k == 0) ? rbyte : (rword[i] | (rbyte << (8 * k)));
            const float2 vc = mul2(zp[i], make_float2(inva, invb));
            cv[h][0] = sr_round(vc.x, 6.0f, wa.y);
            cv[h][1] = sr_round(vc.y, 6.0f, wb.y);
          }
          ca[m2] = e2m1x2(cv[0][0], cv[1][0]);
          cb[m2] = e2m1x2(cv[0][1], cv[1][1]);
        }
        // stage the two half columns' words and (once per column) their scales
        const int c0 = tcol0 + 2 * k;
        *reinterpret_cast<uint32_t*>(cstage + rb * 2048 + stage_col(c0) * 8 + 4 * rh) = pack4(ca[0], ca[1], ca[2], ca[3]);
        *reinterpret_cast<uint32_t*>(cstage + rb * 2048 + stage_col(c0 + 1) * 8 + 4 * rh) =
            pack4(cb[0], cb[1], cb[2], cb[3]);
        if (rh == 0) {
          sstage[stage_col(c0) * 4 + rb] = (uint8_t)ea;
          sstage[stage_col(c0 + 1) * 4 + rb] = (uint8_t)eb;
        }
      }
      if (cols_in) {
        uint8_t* qr = a.q_row + grow0 * hN + gcol0 / 2;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (grow0 + i < M) *reinterpret_cast<uint32_t*>(qr + i * hN) = rword[i];
        if (ch == 0) {
          uint8_t* sr = a.s_row + (a.sf_swz ? tile::sf_swz_off(grow0, gcol0 / 16, (sN + 3) / 4) : grow0 * sN + gcol0 / 16);
          const int64_t sr_step = a.sf_swz ? 16 : sN;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (grow0 + i < M) sr[i * sr_step] = (uint8_t)e_r[i];
        }
      }
    } else {
      // ---- rowwise copy: patch row by patch row
      if (ROW) {
        uint8_t* qr = a.q_row + grow0 * hN + gcol0 / 2;
        uint8_t* sr = a.s_row + (a.sf_swz ? tile::sf_swz_off(grow0, gcol0 / 16, (sN + 3) / 4) : grow0 * sN + gcol0 / 16);
        const int64_t sr_step = a.sf_swz ? 16 : sN;
        const uint64_t ctr0 = a.ctr_off + (uint64_t)grow0 * (uint64_t)N + (uint64_t)gcol0;
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
          // a3: patch row i (eight bf16 values, one 16-byte load)
          uint32_t w4[4];
          {
            const uint4 q = *reinterpret_cast<const uint4*>(pbase + i * 128 + ((pc ^ i) << 4));
            w4[0] = q.x;
            w4[1] = q.y;
            w4[2] = q.z;
            w4[3] = q.w;
          }
          float z[8];
          float bmax;
          if (kRhtRow) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = bf16x2_to_f32x2(w4[k] ^ rht_mask_row(signs, 4 * ch + k));
              z[2 * k] = f.x;
              z[2 * k + 1] = f.y;
            }
            wht8(z);
            bmax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
              const float2 th = make_float2(__shfl_xor_sync(kFull, z[j], 1), __shfl_xor_sync(kFull, z[j + 1], 1));
              const float2 y = last_stage(make_float2(z[j], z[j + 1]), th, ch != 0);
              z[j] = y.x;
              z[j + 1] = y.y;
              bmax = fmaxf(bmax, fmaxf(fabsf(y.x), fabsf(y.y)));
            }
            bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, 1));
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = bf16x2_to_f32x2(w4[k]);
              z[2 * k] = f.x;
              z[2 * k + 1] = f.y;
            }
            uint32_t m = absmax_bf16x2(absmax_bf16x2(w4[0], w4[1]), absmax_bf16x2(w4[2], w4[3]));
            m = absmax_bf16x2(m, __shfl_xor_sync(kFull, m, 1)) & 0x7FFF7FFFu;
            bmax = fmaxf(bf16_lo(m), bf16_hi(m));
          }
          uint32_t e6, e4;
          block_bytes<Q46>(bmax, scR, e6, e4);
          uint32_t sw[8];
          if (SR) {
            const uint64_t ci = ctr0 + (uint64_t)i * (uint64_t)N;
#pragma unroll
            for (int j = 0; j < 8; ++j) sw[j] = words_of(ci + (uint64_t)j, a.sr_k0, a.sr_k1).x;
          }
          uint32_t code, e;
          if (!Q46) {
            float v[8];
            scale8<SR>(z, scR.tbl[e6].y, e6, 6.0f, sw, v);
            code = e2m1x8(v);
            e = e6;
          } else {
            uint32_t c6, c4;
            float s6 = cand8<SR, SEL>(z, e6, scR.tbl[e6], 6.0f, sw, c6);
            float s4 = cand8<SR, SEL>(z, e4, scR.tbl[e4], 4.0f, sw, c4);
            s6 = err_combine(s6, __shfl_xor_sync(kFull, s6, 1), SEL);
            s4 = err_combine(s4, __shfl_xor_sync(kFull, s4, 1), SEL);
            const bool four = s4 < s6;  // strictly lower error: keep the max-4 candidate
            code = four ? c4 : c6;
            e = four ? e4 : e6;
          }
          if (cols_in && grow0 + i < M) {
            *reinterpret_cast<uint32_t*>(qr + i * hN) = code;
            if (ch == 0) sr[i * sr_step] = (uint8_t)e;
          }
        }
      }
      // ---- columnwise copy: patch column pair by column pair
      if (COL) {
        const uint64_t ctr0 = a.ctr_off + (uint64_t)grow0 * (uint64_t)N + (uint64_t)gcol0;
        // Column pairs 2g', 2g'+1 come from one 8-byte load per patch row.
        // Lanes 8-15 and 24-31 take the two groups in the other order, so a
        // half warp reads 16 different 8-byte slots (no bank conflict); the
        // lanes sharing a column block (l, l^16) keep the same order.
        const int rot = (lane >> 3) & 1;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          const int gg = g ^ rot;
          uint32_t w8[8][2];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint2 q = *reinterpret_cast<const uint2*>(pbase + i * 128 + ((pc ^ i) << 4) + 8 * gg);
            w8[i][0] = q.x;
            w8[i][1] = q.y;
          }
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
          const int k = 2 * gg + hk;  // column pair of the patch
          float2 zp[8];
          float ba, bb;
          uint32_t wk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) wk[i] = w8[i][hk];
          if (kRhtCol) {
#pragma unroll
            for (int i = 0; i < 8; ++i) zp[i] = bf16x2_to_f32x2(wk[i] ^ rht_mask_col(signs, 8 * rh + i));
            wht8_x2(zp);
            ba = 0.0f;
            bb = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 th = make_float2(__shfl_xor_sync(kFull, zp[i].x, 16), __shfl_xor_sync(kFull, zp[i].y, 16));
              zp[i] = last_stage(zp[i], th, rh != 0);
              ba = fmaxf(ba, fabsf(zp[i].x));
              bb = fmaxf(bb, fabsf(zp[i].y));
            }
            ba = fmaxf(ba, __shfl_xor_sync(kFull, ba, 16));
            bb = fmaxf(bb, __shfl_xor_sync(kFull, bb, 16));
          } else {
            uint32_t m = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              zp[i] = bf16x2_to_f32x2(wk[i]);
              m = absmax_bf16x2(m, wk[i]);
            }
            m = absmax_bf16x2(m, __shfl_xor_sync(kFull, m, 16)) & 0x7FFF7FFFu;
            ba = bf16_lo(m);
            bb = bf16_hi(m);
          }
          uint32_t e6a, e4a, e6b, e4b;
          block_bytes<Q46>(ba, scC, e6a, e4a);
          block_bytes<Q46>(bb, scC, e6b, e4b);
          uint32_t swa[8], swb[8];
          if (SR) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint64_t ci = ctr0 + (uint64_t)i * (uint64_t)N + (uint64_t)(2 * k);
              swa[i] = words_of(ci, a.sr_k0, a.sr_k1).y;
              swb[i] = words_of(ci + 1u, a.sr_k0, a.sr_k1).y;
            }
          }
          uint2 codes;
          uint32_t ea, eb;
          if (!Q46) {
            float2 v[8];
            scale8x2<SR>(zp, scC.tbl[e6a].y, scC.tbl[e6b].y, e6a, e6b, 6.0f, swa, swb, v);
            codes = encode8x2(v);
            ea = e6a;
            eb = e6b;
          } else {
            uint2 c6, c4;
            float2 s6 = cand8x2<SR, SEL>(zp, e6a, e6b, scC.tbl[e6a], scC.tbl[e6b], 6.0f, swa, swb, c6);
            float2 s4 = cand8x2<SR, SEL>(zp, e4a, e4b, scC.tbl[e4a], scC.tbl[e4b], 4.0f, swa, swb, c4);
            s6.x = err_combine(s6.x, __shfl_xor_sync(kFull, s6.x, 16), SEL);
            s6.y = err_combine(s6.y, __shfl_xor_sync(kFull, s6.y, 16), SEL);
            s4.x = err_combine(s4.x, __shfl_xor_sync(kFull, s4.x, 16), SEL);
            s4.y = err_combine(s4.y, __shfl_xor_sync(kFull, s4.y, 16), SEL);
            const bool fa = s4.x < s6.x, fb = s4.y < s6.y;
            codes = make_uint2(fa ? c4.x : c6.x, fb ? c4.y : c6.y);
            ea = fa ? e4a : e6a;
            eb = fb ? e4b : e6b;
          }
          const int c0 = tcol0 + 2 * k;
          *reinterpret_cast<uint32_t*>(cstage + rb * 2048 + stage_col(c0) * 8 + 4 * rh) = codes.x;
          *reinterpret_cast<uint32_t*>(cstage + rb * 2048 + stage_col(c0 + 1) * 8 + 4 * rh) = codes.y;
          if (rh == 0) {
            sstage[stage_col(c0) * 4 + rb] = (uint8_t)ea;
            sstage[stage_col(c0 + 1) * 4 + rb] = (uint8_t)eb;
          }
          }
        }
      }
    }
    __syncthreads();  // tile buffer free for the next copy; staging complete
    if (COL) write_col_outputs(cstage, sstage, a.q_col, a.s_col, M, N, tc, tid, a.sf_swz != 0);
  }
}

template <bool ROW, bool COL, bool Q46, bool SR, int SEL, int RHT, bool NOCOPY = false>
cudaError_t launch(const QuantArgs& a, cudaStream_t s) {
  auto kern = quant1d_kernel<ROW, COL, Q46, SR, SEL, RHT, NOCOPY>;
  // once per device: opt in to the dynamic shared memory and size the
  // persistent grid from the occupancy
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kBlockThreads, kSmemBytes, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  // persistent grid: every resident CTA slot, or one CTA per tile if fewer
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTN - 1) / kTN);
  int64_t g = ntiles < cap ? ntiles : cap;
  if (g < 1) g = 1;
  CUtensorMap xmap;
  const cudaError_t me = make_tile_map(&xmap, a.x, a.M, a.N, a.ld);
  if (me != cudaSuccess) return me;
  kern<<<(unsigned)g, kBlockThreads, kSmemBytes, s>>>(a, xmap);
  return cudaGetLastError();
}

template <bool ROW, bool COL, bool Q46, int SEL, int RHT>
cudaError_t launch_sr(const QuantArgs& a, bool sr, cudaStream_t s) {
  return sr ? launch<ROW, COL, Q46, true, SEL, RHT>(a, s) : launch<ROW, COL, Q46, false, SEL, RHT>(a, s);
}

// All row/column/SR/RHT combinations of one (4/6, selection rule) pair.
template <bool Q46, int SEL>
cudaError_t launch_family(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s) {
  const int rht = (a.rht_row ? 1 : 0) | (a.rht_col ? 2 : 0);
  if (row && col) {
    switch (rht) {
      case 0: return launch_sr<true, true, Q46, SEL, 0>(a, sr, s);
      case 1: return launch_sr<true, true, Q46, SEL, 1>(a, sr, s);
      case 2: return launch_sr<true, true, Q46, SEL, 2>(a, sr, s);
      default: return launch_sr<true, true, Q46, SEL, 3>(a, sr, s);
    }
  }
  if (row) return rht ? launch_sr<true, false, Q46, SEL, 1>(a, sr, s) : launch_sr<true, false, Q46, SEL, 0>(a, sr, s);
  return rht ? launch_sr<false, true, Q46, SEL, 2>(a, sr, s) : launch_sr<false, true, Q46, SEL, 0>(a, sr, s);
}

}  // namespace q1d
}  // namespace nvfp4
