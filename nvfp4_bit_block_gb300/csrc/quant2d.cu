// quant2d.cu -- NVFP4 quantization with 16x16 2D block scales (weights).
//
// "Pretraining Large Language Models with NVFP4" section 2c: one scale per
// 16x16 tile shared by the forward (rowwise) and the transposed (columnwise)
// copy, so both copies hold the same quantized weight.  Every element is
// quantized once and its code is packed into both layouts, so C's codes are
// exactly the transpose of R's.  With 4/6 the block is scored at maximum 6
// and 4 over all 256 elements ("Four Over Six (4/6)" technical summary,
// Methodology).
//
// Persistent CTAs stream 64 x 256 tiles into double-buffered shared memory
// with TMA (four 64 x 64 boxes, 128-byte swizzle, mbarrier completion with a
// bounded wait), as the 1D kernel does.  Four threads share a 16x16 block,
// each holding an 8 x 8 patch: lane bit 0 picks the column half, lane bit 4
// the row half, so the block max and the 4/6 sums combine with two shuffles
// (xor 1, xor 16).  A warp covers 16 rows x 128 columns; the CTA's 8 warps
// cover the tile.  Each element is encoded once: a patch row's eight codes
// are one rowwise word, and the columnwise bytes (two rows of one column)
// come from interleaving the nibbles of two row words and a 4 x 4 byte
// transpose.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tile_pipeline.cuh"
#include "tma.cuh"

namespace nvfp4 {
namespace {

using tile::kTM;
using tile::kTN;
constexpr int kBlockThreads = 256;

// Philox word 0 of the eight elements (r, c .. c+7) (counter = element index).
__device__ __forceinline__ void words0_of8(const QuantArgs& a, int64_t r, int64_t c, uint32_t* w) {
  philox_group_w01<8, false>(a.ctr_off + (uint64_t)r * (uint64_t)a.N + (uint64_t)c, 1u, a.sr_k0, a.sr_k1, w,
                             nullptr);
}

// Scaled (and, for SR, rounded) value of one element at block scale s.
template <bool SR>
__device__ __forceinline__ float scaled(float z, const BlockScale& s, float Q, uint32_t w) {
  float v = __fmul_rn(z, s.inv);
  if (SR) return sr_round(v, Q, w);
  if (Q == 4.0f && max4_needs_clamp(s.e)) v = fminf(fmaxf(v, -4.0f), 4.0f);
  return v;
}

// Row i (0..7) of this thread's 8 x 8 patch as eight floats.  `pbase` is the
// patch's box plus its first row (a multiple of 8), so with the 128-byte
// swizzle the patch's chunk c of row i sits at (c ^ i) * 16.
__device__ __forceinline__ void patch_row(const uint8_t* pbase, int c, int i, float* z) {
  const uint4 q = *reinterpret_cast<const uint4*>(pbase + i * 128 + ((c ^ i) << 4));
  const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = bf16x2_to_f32x2(wd[k]);
    z[2 * k] = f.x;
    z[2 * k + 1] = f.y;
  }
}

// One 4/6 candidate on one patch row: the 8 codes at scale s (maximum Q) and
// this row part's score -- err = z - val*d rounded once, |err| (MAE, MAXERR)
// or err*err (MSE), combined as the perfect binary tree over the 8 values in
// order.  The row's two column halves, the 8 rows of a half and the two halves
// are combined by the caller, so the score of the 16x16 block is the same
// tree over its 256 values in row-major order.
template <bool SR, int SEL>
__device__ __forceinline__ float cand8(const float* z, const BlockScale& s, float Q, const uint32_t* w,
                                       uint32_t& codes) {
  const float2 inv2 = make_float2(s.inv, s.inv);
  const float2 nd = make_float2(-s.d, -s.d);
  float v[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 r = mul2(make_float2(z[2 * j], z[2 * j + 1]), inv2);
    v[2 * j] = r.x;
    v[2 * j + 1] = r.y;
  }
  if (SR) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = sr_round(v[j], Q, w[j]);
  } else if (Q == 4.0f && max4_needs_clamp(s.e)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fminf(fmaxf(v[j], -4.0f), 4.0f);
  }
  uint32_t h[4];
  codes = e2m1x8_enc_dec(v, h);
  float t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 err = fma2(f16x2_to_f32x2(h[k]), nd, make_float2(z[2 * k], z[2 * k + 1]));
    if (SEL == kSelMSE) {
      const float2 sq = mul2(err, err);
      t[k] = __fadd_rn(sq.x, sq.y);
    } else if (SEL == kSelMax) {
      t[k] = fmaxf(fabsf(err.x), fabsf(err.y));
    } else {
      t[k] = __fadd_rn(fabsf(err.x), fabsf(err.y));
    }
  }
  return err_combine(err_combine(t[0], t[1], SEL), err_combine(t[2], t[3], SEL), SEL);
}

// Byte m of each of w[0..3] gathered into output word m (a 4 x 4 byte transpose).
__device__ __forceinline__ void transpose4x4(const uint32_t* w, uint32_t* t) {
  const uint32_t a_lo = __byte_perm(w[0], w[1], 0x5140), a_hi = __byte_perm(w[0], w[1], 0x7362);
  const uint32_t b_lo = __byte_perm(w[2], w[3], 0x5140), b_hi = __byte_perm(w[2], w[3], 0x7362);
  t[0] = __byte_perm(a_lo, b_lo, 0x5410);
  t[1] = __byte_perm(a_lo, b_lo, 0x7632);
  t[2] = __byte_perm(a_hi, b_hi, 0x5410);
  t[3] = __byte_perm(a_hi, b_hi, 0x7632);
}

template <bool ROW, bool COL, bool Q46, bool SR, int SEL>
__global__ void __launch_bounds__(kBlockThreads, SR ? 2 : 3)
    quant2d_kernel(const QuantArgs a, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bufs = smem;                                  // 2 x 32 KB tiles (1024-aligned)
  uint8_t* cstage = smem + 2 * tile::kTileBytes;  // padded layouts (lanes hold columns 8 apart)
  uint8_t* sstage = cstage + tile::kCStagePadBytes;
  const uint32_t bar0 = tile::smem_u32(sstage + tile::kSStagePadBytes), bar1 = bar0 + 8;

  const float den = Q46 ? kAlphaDen46 : kAlphaDen;
  const float A = a.amax[0];
  const float alpha = __fdiv_rn(A, den);
  const int st = amax_status(A);
  const bool misaligned = (tile::smem_u32(smem) & 1023u) != 0u;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha;
    a.alpha[1] = __fdiv_rn(a.amax[1], den);
    if (st && a.status) *a.status = st;
    if (misaligned && !st && a.status) *a.status = kStatusPipeline;
  }
  if (st || misaligned) return;

  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ch = lane & 1, bcol = (lane >> 1) & 7, rh = lane >> 4;
  const int rb = warp >> 1;                                // row block of this warp
  const int tcol0 = 128 * (warp & 1) + 16 * bcol + 8 * ch; // first tile column of this thread
  const int trow0 = 16 * rb + 8 * rh;                      // first tile row of this thread
  const int pc = (tcol0 & 63) >> 3;                        // the patch's 16-byte chunk within its box
  const uint32_t poff = (tcol0 >> 6) * 8192 + trow0 * 128; // the patch's box and first row
  const int64_t hN = N / 2, sN = N / 16;
  if (tid == 0) {
    tma::mbar_init(bar0, 1);
    tma::mbar_init(bar1, 1);
    tma::fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int b, const tile::Coord& c) {
    const uint32_t bar = b ? bar1 : bar0;
    tma::arrive_expect_tx(bar, tile::kTileBytes);
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
      if (tid == 0) {
        if (a.status) atomicExch(a.status, kStatusPipeline);
        tma::wait(b ? bar1 : bar0, parity);
        if (w.next().valid()) tma::wait(b ? bar0 : bar1, ((it + 1) >> 1) & 1);
      }
      return;
    }
    const tile::Coord tc = w.coord();
    const int64_t grow0 = tc.R0 + trow0, gcol0 = tc.C0 + tcol0;
    // a block is valid when its 16 rows and 16 columns lie inside the tensor
    const bool valid = (tc.R0 + 16 * rb < M) && (tc.C0 + (tcol0 & ~15) < N);
    const uint8_t* pbase = buf + poff;

    // a5: block maximum over 256 values
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 q = *reinterpret_cast<const uint4*>(pbase + i * 128 + ((pc ^ i) << 4));
      m2 = absmax_bf16x2(m2, absmax_bf16x2(absmax_bf16x2(q.x, q.y), absmax_bf16x2(q.z, q.w)));
    }
    m2 &= 0x7FFF7FFFu;
    float bmax = fmaxf(bf16_lo(m2), bf16_hi(m2));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 1));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 16));

    // a9: a patch row's code word goes to R directly, and each pair of rows
    // becomes C bytes (column j = 2m: byte m of lo; j = 2m+1: byte m of hi;
    // the first row in the low nibble)
    uint32_t lo[4], hi[4];
    uint8_t* qr = a.q_row + grow0 * hN + gcol0 / 2;
    auto store_row = [&](int i, uint32_t c) {
      if (ROW && valid) *reinterpret_cast<uint32_t*>(qr + i * hN) = c;
    };
    auto interleave = [&](int p2, uint32_t c0, uint32_t c1) {
      lo[p2] = (c0 & 0x0F0F0F0Fu) | ((c1 & 0x0F0F0F0Fu) << 4);
      hi[p2] = ((c0 >> 4) & 0x0F0F0F0Fu) | (c1 & 0xF0F0F0F0u);
    };

    // a6-a8: each element is scaled and rounded once per candidate
    BlockScale s = block_scale(bmax, alpha, 6.0f);
    if (Q46) {  // both candidates scored in one pass; both candidates' code rows kept
      const BlockScale s4 = block_scale(bmax, alpha, 4.0f);
      uint32_t code6[8], code4[8];
      float r6[8], r4[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float z[8];
        patch_row(pbase, pc, i, z);
        uint32_t w[8];
        if (SR) words0_of8(a, grow0 + i, gcol0, w);
        const float p6 = cand8<SR, SEL>(z, s, 6.0f, w, code6[i]);
        const float p4 = cand8<SR, SEL>(z, s4, 4.0f, w, code4[i]);
        r6[i] = err_combine(p6, __shfl_xor_sync(0xFFFFFFFFu, p6, 1), SEL);
        r4[i] = err_combine(p4, __shfl_xor_sync(0xFFFFFFFFu, p4, 1), SEL);
      }
      auto tree8 = [](const float* r) {
        return err_combine(err_combine(err_combine(r[0], r[1], SEL), err_combine(r[2], r[3], SEL), SEL),
                           err_combine(err_combine(r[4], r[5], SEL), err_combine(r[6], r[7], SEL), SEL), SEL);
      };
      const float h6 = tree8(r6), h4 = tree8(r4);
      const float sc6 = err_combine(h6, __shfl_xor_sync(0xFFFFFFFFu, h6, 16), SEL);
      const float sc4 = err_combine(h4, __shfl_xor_sync(0xFFFFFFFFu, h4, 16), SEL);
      const bool four = sc4 < sc6;  // strictly lower error: keep the max-4 candidate
      if (four) s = s4;
#pragma unroll
      for (int p2 = 0; p2 < 4; ++p2) {
        const uint32_t c0 = four ? code4[2 * p2] : code6[2 * p2], c1 = four ? code4[2 * p2 + 1] : code6[2 * p2 + 1];
        store_row(2 * p2, c0);
        store_row(2 * p2 + 1, c1);
        interleave(p2, c0, c1);
      }
    } else {
#pragma unroll
      for (int p2 = 0; p2 < 4; ++p2) {
        uint32_t code[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 2 * p2 + h;
          float z[8], v[8];
          patch_row(pbase, pc, i, z);
          if (SR) {
            uint32_t w[8];
            words0_of8(a, grow0 + i, gcol0, w);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = scaled<true>(z[j], s, 6.0f, w[j]);
          } else {
            const float2 inv2 = make_float2(s.inv, s.inv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 r = mul2(make_float2(z[2 * j], z[2 * j + 1]), inv2);
              v[2 * j] = r.x;
              v[2 * j + 1] = r.y;
            }
          }
          code[h] = e2m1x8(v);
          store_row(i, code[h]);
        }
        interleave(p2, code[0], code[1]);
      }
    }
    if (COL) {
      uint32_t tl[4], th[4];
      transpose4x4(lo, tl);
      transpose4x4(hi, th);
      // the thread's 8 columns lie inside one 16-column group: one pad offset
      uint8_t* cs = cstage + tile::cstage_off_pad(rb, tcol0) + 4 * rh;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        *reinterpret_cast<uint32_t*>(cs + (2 * m) * 8) = tl[m];
        *reinterpret_cast<uint32_t*>(cs + (2 * m + 1) * 8) = th[m];
      }
      if (rh == 0) {
        uint8_t* ss = sstage + tile::sstage_off_pad(tcol0) + rb;  // 8 columns, one 8-column group
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[4 * j] = (uint8_t)s.e;
      }
    }
    if (ROW && valid && ch == 0) {
      // 8 consecutive rows from a multiple of 8: 16 bytes apart in the tiled layout
      uint8_t* sr = a.s_row + (a.sf_swz ? tile::sf_swz_off(grow0, gcol0 / 16, (sN + 3) / 4) : grow0 * sN + gcol0 / 16);
      const int64_t sr_step = a.sf_swz ? 16 : sN;
#pragma unroll
      for (int i = 0; i < 8; ++i) sr[i * sr_step] = (uint8_t)s.e;
    }
    __syncthreads();  // tile buffer free for the next copy; staging complete
    if (COL) tile::write_col_outputs<true>(cstage, sstage, a.q_col, a.s_col, M, N, tc, tid, a.sf_swz != 0);
  }
}

template <bool ROW, bool COL, bool Q46, bool SR, int SEL>
cudaError_t launch(const QuantArgs& a, cudaStream_t st) {
  constexpr int kSmem = 2 * tile::kTileBytes + tile::kCStagePadBytes + tile::kSStagePadBytes + 16;  // + 2 barriers
  auto kern = quant2d_kernel<ROW, COL, Q46, SR, SEL>;
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kBlockThreads, kSmem, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTN - 1) / kTN);
  int64_t grid = ntiles < cap ? ntiles : cap;
  if (grid < 1) grid = 1;
  CUtensorMap xmap;
  const cudaError_t me = make_tile_map(&xmap, a.x, a.M, a.N, a.ld);
  if (me != cudaSuccess) return me;
  kern<<<(unsigned)grid, kBlockThreads, kSmem, st>>>(a, xmap);
  return cudaGetLastError();
}

template <bool ROW, bool COL, bool Q46, int SEL>
cudaError_t launch_sr(const QuantArgs& a, bool sr, cudaStream_t st) {
  return sr ? launch<ROW, COL, Q46, true, SEL>(a, st) : launch<ROW, COL, Q46, false, SEL>(a, st);
}

template <bool ROW, bool COL>
cudaError_t launch_rc(const QuantArgs& a, bool q46, bool sr, cudaStream_t st) {
  if (!q46) return launch_sr<ROW, COL, false, kSelMAE>(a, sr, st);
  if (a.sel == kSelMSE) return launch_sr<ROW, COL, true, kSelMSE>(a, sr, st);
  if (a.sel == kSelMax) return launch_sr<ROW, COL, true, kSelMax>(a, sr, st);
  return launch_sr<ROW, COL, true, kSelMAE>(a, sr, st);
}

}  // namespace

cudaError_t launch_quant2d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t st) {
  if (row && col) return launch_rc<true, true>(a, q46, sr, st);
  if (row) return launch_rc<true, false>(a, q46, sr, st);
  return launch_rc<false, true>(a, q46, sr, st);
}

}  // namespace nvfp4
