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
// Persistent CTAs stream 64 x 256 tiles through double-buffered shared memory
// (tile_pipeline.cuh).  Four threads share a 16x16 block, each holding 8 rows
// x 8 columns: lane bit 0 picks the column half, lane bit 4 the row half, so
// the block max and the 4/6 sums combine with two shuffles (xor 1, xor 16).
// A warp covers 16 rows x 128 columns; the CTA's 8 warps cover the tile.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tile_pipeline.cuh"

namespace nvfp4 {
namespace {

using tile::kTM;
using tile::kTN;
constexpr int kBlockThreads = 256;

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

// This thread's 8 values of row `lr` (0..7 within its row half).
__device__ __forceinline__ void row8(const uint8_t* buf, int trow, int chunk, float* z) {
  const uint4 q = *reinterpret_cast<const uint4*>(buf + trow * tile::kRowBytes + tile::swz(chunk) * 16);
  z[0] = bf16_lo(q.x); z[1] = bf16_hi(q.x);
  z[2] = bf16_lo(q.y); z[3] = bf16_hi(q.y);
  z[4] = bf16_lo(q.z); z[5] = bf16_hi(q.z);
  z[6] = bf16_lo(q.w); z[7] = bf16_hi(q.w);
}

// 4/6 score of the 16x16 block at scale s: per row a tree over this lane's 8
// columns plus the column partner's, then a tree over this row half's 8 rows,
// then the two row halves.  Same order as a perfect binary tree over the 256
// elements in row-major order.
template <bool SR>
__device__ __forceinline__ float block_score(const uint8_t* buf, int trow0, int chunk, const BlockScale& s,
                                             float Q, const QuantArgs& a, int64_t grow0, int64_t gcol0, int sel) {
  float rows[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float z[8], v[8];
    row8(buf, trow0 + i, chunk, z);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = scaled<SR>(z[j], s, Q, SR ? word0_of(a, grow0 + i, gcol0 + j) : 0u);
    const float part = score8(z, e2m1x8(v), s.d, sel);
    rows[i] = err_combine(part, __shfl_xor_sync(0xFFFFFFFFu, part, 1), sel);
  }
  const float h = err_combine(err_combine(err_combine(rows[0], rows[1], sel), err_combine(rows[2], rows[3], sel), sel),
                              err_combine(err_combine(rows[4], rows[5], sel), err_combine(rows[6], rows[7], sel), sel),
                              sel);
  return err_combine(h, __shfl_xor_sync(0xFFFFFFFFu, h, 16), sel);
}

template <bool ROW, bool COL, bool Q46, bool SR>
__global__ void __launch_bounds__(kBlockThreads) quant2d_kernel(const QuantArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* bufs = smem;
  uint8_t* cstage = smem + 2 * tile::kTileBytes;
  uint8_t* sstage = cstage + tile::kCStageBytes;

  const float den = Q46 ? kAlphaDen46 : kAlphaDen;
  const float A = a.amax[0];
  const float alpha = __fdiv_rn(A, den);
  const int st = amax_status(A);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha;
    a.alpha[1] = __fdiv_rn(a.amax[1], den);
    if (st && a.status) *a.status = st;
  }
  if (st) return;

  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ch = lane & 1, bcol = (lane >> 1) & 7, rh = lane >> 4;
  const int rb = warp >> 1;                                // row block of this warp
  const int tcol0 = 128 * (warp & 1) + 16 * bcol + 8 * ch; // first tile column of this thread
  const int chunk = tcol0 >> 3;
  const int trow0 = 16 * rb + 8 * rh;                      // first tile row of this thread

  tile::Walker w;
  w.init(M, N);
  if (w.valid()) tile::load_async<kBlockThreads>(bufs, a.x, M, N, a.ld, w.coord(), tid);
  tile::commit();
  for (int it = 0; w.valid(); w = w.next(), ++it) {
    uint8_t* buf = bufs + (it & 1) * tile::kTileBytes;
    const tile::Walker wn = w.next();
    if (wn.valid())
      tile::load_async<kBlockThreads>(bufs + ((it + 1) & 1) * tile::kTileBytes, a.x, M, N, a.ld, wn.coord(), tid);
    tile::commit();
    tile::wait_all_but_one();
    __syncthreads();
    const tile::Coord tc = w.coord();
    const int64_t grow0 = tc.R0 + trow0, gcol0 = tc.C0 + tcol0;
    // a block is valid when its 16 rows and 16 columns lie inside the tensor
    const bool valid = (tc.R0 + 16 * rb < M) && (tc.C0 + (tcol0 & ~15) < N);

    // a5: block maximum over 256 values
    uint32_t m2 = 0u;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const uint4 q = *reinterpret_cast<const uint4*>(buf + (trow0 + i) * tile::kRowBytes + tile::swz(chunk) * 16);
      m2 = absmax_bf16x2(m2, absmax_bf16x2(absmax_bf16x2(q.x, q.y), absmax_bf16x2(q.z, q.w)));
    }
    m2 &= 0x7FFF7FFFu;
    float b = fmaxf(bf16_lo(m2), bf16_hi(m2));
    b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
    b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 16));

    BlockScale s = block_scale(b, alpha, 6.0f);
    float Q = 6.0f;
    if (Q46) {
      const BlockScale s4 = block_scale(b, alpha, 4.0f);
      const float sc6 = block_score<SR>(buf, trow0, chunk, s, 6.0f, a, grow0, gcol0, a.sel);
      const float sc4 = block_score<SR>(buf, trow0, chunk, s4, 4.0f, a, grow0, gcol0, a.sel);
      if (sc4 < sc6) {
        s = s4;
        Q = 4.0f;
      }
    }

    // a7 + a9: each element once, packed rowwise (pairs along a row, stored
    // directly) and columnwise (pairs along a column, staged)
    uint32_t cq[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
    for (int i = 0; i < 8; i += 2) {
      float z0[8], z1[8], v0[8], v1[8];
      row8(buf, trow0 + i, chunk, z0);
      row8(buf, trow0 + i + 1, chunk, z1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v0[j] = scaled<SR>(z0[j], s, Q, SR ? word0_of(a, grow0 + i, gcol0 + j) : 0u);
        v1[j] = scaled<SR>(z1[j], s, Q, SR ? word0_of(a, grow0 + i + 1, gcol0 + j) : 0u);
      }
      if (ROW && valid) {
        *reinterpret_cast<uint32_t*>(a.q_row + (grow0 + i) * (N / 2) + gcol0 / 2) = e2m1x8(v0);
        *reinterpret_cast<uint32_t*>(a.q_row + (grow0 + i + 1) * (N / 2) + gcol0 / 2) = e2m1x8(v1);
      }
      if (COL) {
#pragma unroll
        for (int j = 0; j < 8; ++j) cq[j] |= e2m1x2(v0[j], v1[j]) << (4 * i);
      }
    }
    if (COL) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint32_t*>(cstage + rb * (kTN * 8) + (tcol0 + j) * 8 + 4 * rh) = cq[j];
      if (rh == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) sstage[(tcol0 + j) * 4 + rb] = (uint8_t)s.e;
      }
    }
    if (ROW && valid && ch == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) a.s_row[(grow0 + i) * (N / 16) + gcol0 / 16] = (uint8_t)s.e;
    }
    __syncthreads();
    if (COL) tile::write_col_outputs(cstage, sstage, a.q_col, a.s_col, M, N, tc, tid);
  }
}

template <bool ROW, bool COL, bool Q46, bool SR>
cudaError_t launch(const QuantArgs& a, cudaStream_t st) {
  constexpr int kSmem = 2 * tile::kTileBytes + tile::kCStageBytes + tile::kSStageBytes;
  auto kern = quant2d_kernel<ROW, COL, Q46, SR>;
  static int grid_cap[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int cap = (dev >= 0 && dev < 64) ? grid_cap[dev] : 0;
  if (cap == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBlockThreads, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cap = (per_sm > 0 ? per_sm : 1) * sms;
    if (dev >= 0 && dev < 64) grid_cap[dev] = cap;
  }
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTN - 1) / kTN);
  int64_t grid = ntiles < cap ? ntiles : cap;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kBlockThreads, kSmem, st>>>(a);
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
