#pragma once
// quant1d_sr_kernel.cuh -- rowwise + columnwise NVFP4 quantization with 1x16
// blocks and stochastic rounding on both copies, from one Philox4x32-10 call
// per element (word 0 rounds the element's rowwise code, word 1 its
// columnwise code).
//
// Both roundings of an element happen in one thread.  Per 64 x 256 tile:
//   - a rowwise pre-pass finds every rowwise block's maximum and scale byte,
//     writes the byte and keeps the block's reciprocal scale in shared memory;
//   - the columnwise pass gives each thread a column pair over 16 rows (as in
//     quant1d_kernel): it finds the two columnwise scales, draws the 32
//     elements' Philox words and rounds each element twice -- for the
//     columnwise copy with word 1, for the rowwise copy with word 0 and the
//     rowwise block's reciprocal scale.  The two columns of a pair are the
//     two codes of one rowwise byte, so each row yields one finished byte;
//   - the rowwise code bytes (64 rows x 128 bytes) and the columnwise codes
//     are staged in shared memory and written out after the tile.
// Against parking word 1 of every element for a later pass (64 KB of shared
// memory), the staging takes 8 KB, so the tiles are double-buffered, and the
// integer multiplies of Philox and the floating-point work of the roundings
// run interleaved in every warp.  The pre-pass of the next tile and the
// write-out of the current one share a barrier interval: two barriers per
// tile.
//
// Not handled here: a Hadamard transform on the rowwise copy (the pre-pass
// takes plain maxima) and 4/6 (its choice needs a whole rowwise block in one
// thread); quant1d_kernel covers those.
//
// Sources: "Pretraining Large Language Models with NVFP4" sections 2b
// (random Hadamard transform) and 2d (stochastic rounding), "Four Over Six
// (4/6)" technical summary (Problem statement: E2M1 grid and block scaling).
#include <type_traits>

#include "quant1d_common.cuh"

namespace nvfp4 {
namespace q1d {

constexpr int kRStageBytes = kTM * kTN / 2;  // rowwise code bytes of a tile, 8 KB
// Reciprocal scale of rowwise block b (0..15) of tile row r at b * 72 + r:
// the pre-pass's stores from a warp (8 rows x 4 blocks) fall in 32 distinct
// banks, and a columnwise warp's reads (one row, 4 blocks) are broadcasts.
constexpr int kRInvStride = 72;
constexpr int kRInvBytes = (kTN / 16) * kRInvStride * 4;
// Rows of a column pair whose Philox words are drawn together (two calls per
// row in flight per thread).  Two rows measured fastest: 4 and 8 rows hold
// more registers (118-128) for 1-2 % more time.
constexpr int kChunkRows = 2;

// Words 0 and 1 of the counters base + i * stride + h, i = I0..I0+R-1,
// h = 0, 1 (stride < 2^32); p0r1 is the shared second-round product of word
// 0 when all sixteen rows of the column pair share their high word.
template <int I0, int R>
__device__ __forceinline__ void philox_rows(uint64_t base, uint32_t stride, bool shared_hi, uint64_t p0r1,
                                            uint32_t k0, uint32_t k1, uint32_t (&w0)[R][2], uint32_t (&w1)[R][2]) {
  if (shared_hi) {
    const uint32_t lo = (uint32_t)base + (uint32_t)I0 * stride;
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint2 r = philox_w01_shared_hi(lo + (uint32_t)j * stride + (uint32_t)h, p0r1, k0, k1);
        w0[j][h] = r.x;
        w1[j][h] = r.y;
      }
  } else {
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t c = base + (uint64_t)(I0 + j) * stride + (uint64_t)h;
        const uint2 r = philox_w01((uint32_t)c, (uint32_t)(c >> 32), k0, k1);
        w0[j][h] = r.x;
        w1[j][h] = r.y;
      }
  }
}

// f(integral_constant<int, I>) for I = BEGIN, BEGIN + STEP, ... < END.
template <int BEGIN, int END, int STEP, typename F>
__device__ __forceinline__ void static_for(F& f) {
  if constexpr (BEGIN < END) {
    f(std::integral_constant<int, BEGIN>{});
    static_for<BEGIN + STEP, END, STEP>(f);
  }
}

// Write the staged rowwise codes of one tile: thread t writes 16-byte chunk
// t % 8 of tile rows t / 8 and t / 8 + 32 (a row's valid bytes are cols / 2).
// A quarter warp reads one whole 128-byte row, so the reads are free of bank
// conflicts, and a warp's stores cover four whole rows.
__device__ __forceinline__ void write_row_outputs(const uint8_t* rstage, uint8_t* q_row, int64_t hN,
                                                  const tile::Coord& tc, int rows, int cols, int tid) {
  const int c = tid & 7;
  if (16 * c >= cols / 2) return;  // cols / 2 is a multiple of 8; chunks are whole or absent
  const bool half = 16 * c + 8 >= cols / 2;  // only the chunk's first 8 bytes are in the tensor
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = (tid >> 3) + 32 * h;
    if (r >= rows) break;
    const uint4 v = *reinterpret_cast<const uint4*>(rstage + r * 128 + 16 * c);
    uint8_t* dst = q_row + (tc.R0 + r) * hN + tc.C0 / 2 + 16 * c;
    if (!half && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      *reinterpret_cast<uint4*>(dst) = v;
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(v.x, v.y);
      if (!half) *reinterpret_cast<uint2*>(dst + 8) = make_uint2(v.z, v.w);
    }
  }
}

// RHT_COL: Hadamard transform on the columnwise copy.
// NOCOPY (a test instantiation only): arm the tile barriers but issue no copy.
template <bool RHT_COL, bool NOCOPY = false>
__global__ void __launch_bounds__(kBlockThreads, 2)
    quant1d_sr_kernel(const QuantArgs a, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bufs = smem;                                          // 2 x 32 KB tiles (1024-aligned)
  uint8_t* cstage = smem + 2 * tile::kTileBytes;                 // 8 KB
  uint8_t* sstage = cstage + tile::kCStageBytes;                 // 1 KB
  uint8_t* rstage = sstage + tile::kSStageBytes;                 // 8 KB
  float* rinv = reinterpret_cast<float*>(rstage + kRStageBytes);  // 4.5 KB
  // 1/d per scale byte e: rowwise copy tinv[e], columnwise tinv[128 + e]
  // (4-byte entries: lanes reading different bytes share a bank only when
  // the bytes are 32 apart), then the two tile barriers
  float* tinv = rinv + kRInvBytes / 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tinv + 256);
  const uint32_t bar0 = tile::smem_u32(bars), bar1 = tile::smem_u32(bars + 1);

  float alpha_r, alpha_c;
  if (!begin_tensor(a, true, true, kAlphaDen, smem, alpha_r, alpha_c)) return;

  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x;
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
  if (tid == 0) {
    tma::mbar_init(bar0, 1);
    tma::mbar_init(bar1, 1);
    tma::fence_barrier_init();
    if (w.valid()) {
      issue(0, w.coord());
      const tile::Walker wn = w.next();
      if (wn.valid()) issue(1, wn.coord());
    }
  }
  tinv[tid] = scale_entry(tid & 127, (tid >> 7) ? alpha_c : alpha_r).y;
  __syncthreads();  // barriers and tables ready
  if (!w.valid()) return;
  const CopyScales scR = make_scales(alpha_r, nullptr);  // den and 1/den; 1/d comes from tinv
  const CopyScales scC = make_scales(alpha_c, nullptr);
  const uint32_t signs = RHT_COL ? rht_sign_bits(a.rht_k0, a.rht_k1) : 0u;
  const uint32_t k0 = a.sr_k0, k1 = a.sr_k1;
  const uint32_t N32 = (uint32_t)N;

  // Fixed per-thread roles (tile layout and the first two as in quant1d_kernel):
  //  pre-pass   tile row rr = 8*warp + lane/4, blocks rq + 4k (k = 0..3)
  //  columnwise column pair cp_p, row blocks cp_rb0 + 2k (k = 0..1)
  //  write-out  rowwise: tile row tid/4, 32 bytes; columnwise: tile column tid
  const int lane = tid & 31;
  const int rr = 8 * (tid >> 5) + (lane >> 2), rq = lane & 3;
  const uint32_t r_chunk0 = rr * 128 + ((uint32_t)((2 * rq) ^ (lane >> 2)) << 4);  // second chunk: ^ 16
  const int64_t hN = N / 2, sN = N / 16;
  const int cp_p = tid & 127, cp_rb0 = tid >> 7;
  const uint32_t c_base = (cp_p >> 5) * 8192 + (cp_p & 3) * 4;
  const uint32_t c_chunk = (uint32_t)((cp_p & 31) >> 2) << 4;

  // rowwise block maxima of a tile -> scale bytes (written) and 1/d (kept)
  auto prepass = [&](const uint8_t* buf, const tile::Coord& tc) {
    const int rows = (int)((M - tc.R0) < kTM ? (M - tc.R0) : kTM);
    const int cols = (int)((N - tc.C0) < kTN ? (N - tc.C0) : kTN);
    if (rr >= rows) return;
    uint8_t* st = a.s_row + (a.sf_swz ? tile::sf_swz_off(tc.R0 + rr, tc.C0 / 16 + rq, (sN + 3) / 4)
                                      : (tc.R0 + rr) * sN + tc.C0 / 16 + rq);
    const int st_step = a.sf_swz ? 512 : 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (16 * (rq + 4 * k) >= cols) break;
      uint32_t wd[8];
      const uint4 lo = *reinterpret_cast<const uint4*>(buf + k * 8192 + r_chunk0);
      const uint4 hi = *reinterpret_cast<const uint4*>(buf + k * 8192 + (r_chunk0 ^ 16u));
      wd[0] = lo.x; wd[1] = lo.y; wd[2] = lo.z; wd[3] = lo.w;
      wd[4] = hi.x; wd[5] = hi.y; wd[6] = hi.z; wd[7] = hi.w;
      const uint32_t e = scale_byte(block_absmax16(wd), scR.den6, scR.rden6);
      rinv[(rq + 4 * k) * kRInvStride + rr] = tinv[e];
      st[st_step * k] = (uint8_t)e;
    }
  };

  // both copies' codes of column pair p, row block rb (16 rows)
  auto colpass = [&](const uint8_t* buf, const tile::Coord& tc) {
    const int rows = (int)((M - tc.R0) < kTM ? (M - tc.R0) : kTM);
    const int cols = (int)((N - tc.C0) < kTN ? (N - tc.C0) : kTN);
    const int p = cp_p;
    if (2 * p >= cols) return;
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      const int rb = cp_rb0 + 2 * k;
      if (16 * rb >= rows) break;
      uint32_t wd[16];
      const uint8_t* cb = buf + c_base + rb * 2048;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        wd[i] = *reinterpret_cast<const uint32_t*>(cb + i * 128 + (c_chunk ^ ((uint32_t)(i & 7) << 4)));
      // columnwise values and maxima (low half = column 2p, high half = 2p+1)
      float2 y[16];  // with RHT_COL: the transformed columnwise values
      float bm0, bm1;
      if (RHT_COL) {
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = bf16x2_to_f32x2(wd[i] ^ rht_mask_col(signs, i));
        wht16_x2(y);
        bm0 = bm1 = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          y[i] = mul2(y[i], make_float2(0.25f, 0.25f));
          bm0 = fmaxf(bm0, fabsf(y[i].x));
          bm1 = fmaxf(bm1, fabsf(y[i].y));
        }
      } else {
        uint32_t t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = absmax_bf16x2(wd[2 * i], wd[2 * i + 1]);
        const uint32_t m2 =
            absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(t8[0], t8[1]), absmax_bf16x2(t8[2], t8[3])),
                          absmax_bf16x2(absmax_bf16x2(t8[4], t8[5]), absmax_bf16x2(t8[6], t8[7]))) &
            0x7FFF7FFFu;
        bm0 = bf16_lo(m2);
        bm1 = bf16_hi(m2);
      }
      const uint32_t ec0 = scale_byte(bm0, scC.den6, scC.rden6);
      const uint32_t ec1 = scale_byte(bm1, scC.den6, scC.rden6);
      const float2 invc = make_float2(tinv[128 + ec0], tinv[128 + ec1]);
      const float* ri = rinv + (p >> 3) * kRInvStride + 16 * rb;  // row i of the block: ri[i]
      uint8_t* rs = rstage + (16 * rb) * 128 + p;                  // row i: rs[128 * i]
      const uint64_t base = a.ctr_off + (uint64_t)((tc.R0 + 16 * rb) * N + tc.C0 + 2 * p);
      const uint64_t last = base + (uint64_t)15 * N32 + 1u;
      const bool shared_hi = (uint32_t)(base >> 32) == (uint32_t)(last >> 32);
      const uint64_t p0r1 = (uint64_t)0xD2511F53u * ((uint32_t)(base >> 32) ^ k0);
      uint32_t cb0[8], cb1[8];  // columnwise code bytes (rows 2i, 2i+1) of columns 2p and 2p+1
      // rows I0 .. I0 + kChunkRows - 1 of both columns: Philox words, then
      // both roundings of each element
      auto chunk = [&](auto i0c) {
        constexpr int I0 = decltype(i0c)::value;
        uint32_t w0[kChunkRows][2], w1[kChunkRows][2];
        philox_rows<I0, kChunkRows>(base, N32, shared_hi, p0r1, k0, k1, w0, w1);
        float gc0[kChunkRows], gc1[kChunkRows];
#pragma unroll
        for (int j = 0; j < kChunkRows; ++j) {
          const int i = I0 + j;
          const float2 x = bf16x2_to_f32x2(wd[i]);
          float2 yc = x;
          if constexpr (RHT_COL) yc = y[i];
          const float ir = ri[i];
          const float2 vr = mul2(x, make_float2(ir, ir));
          const float2 vc = mul2(yc, invc);
          const float gr0 = sr_round(vr.x, 6.0f, w0[j][0]);
          const float gr1 = sr_round(vr.y, 6.0f, w0[j][1]);
          gc0[j] = sr_round(vc.x, 6.0f, w1[j][0]);
          gc1[j] = sr_round(vc.y, 6.0f, w1[j][1]);
          rs[128 * i] = (uint8_t)e2m1x2(gr0, gr1);
        }
#pragma unroll
        for (int j = 0; j < kChunkRows; j += 2) {
          cb0[(I0 + j) / 2] = e2m1x2(gc0[j], gc0[j + 1]);
          cb1[(I0 + j) / 2] = e2m1x2(gc1[j], gc1[j + 1]);
        }
      };
      static_assert(16 % kChunkRows == 0 && kChunkRows % 2 == 0, "chunks of whole code bytes");
      static_for<0, 16, kChunkRows>(chunk);
      const uint2 c0 = make_uint2(pack4(cb0[0], cb0[1], cb0[2], cb0[3]), pack4(cb0[4], cb0[5], cb0[6], cb0[7]));
      const uint2 c1 = make_uint2(pack4(cb1[0], cb1[1], cb1[2], cb1[3]), pack4(cb1[4], cb1[5], cb1[6], cb1[7]));
      tile::stage_col_pair(cstage, sstage, p, rb, c0, c1, ec0, ec1);
    }
  };

  const bool first = tma::wait(bar0, 0);
  if (!__syncthreads_and(first)) {
    // the first tile did not arrive in time: report it, give the copies in
    // flight one more bounded wait, and stop
    if (tid == 0) {
      if (a.status) atomicExch(a.status, kStatusPipeline);
      tma::wait(bar0, 0);
      if (w.next().valid()) tma::wait(bar1, 0);
    }
    return;
  }
  prepass(bufs, w.coord());
  for (int it = 0;; ++it) {
    const int b = it & 1;
    const tile::Coord tc = w.coord();
    __syncthreads();  // rowwise scales of this tile ready; the last tile's staging written out
    colpass(bufs + b * tile::kTileBytes, tc);
    const tile::Walker wn = w.next();
    const bool more = wn.valid();
    const bool arrived = more ? tma::wait(b ? bar0 : bar1, ((it + 1) >> 1) & 1) : true;
    if (!__syncthreads_and(arrived)) {
      if (tid == 0) {
        if (a.status) atomicExch(a.status, kStatusPipeline);
        tma::wait(b ? bar0 : bar1, ((it + 1) >> 1) & 1);
      }
      return;
    }
    // every thread is done with buffer b: it takes the tile after the next
    if (tid == 0) {
      const tile::Walker wnn = wn.next();
      if (more && wnn.valid()) issue(b, wnn.coord());
    }
    if (more) prepass(bufs + (b ^ 1) * tile::kTileBytes, wn.coord());
    {
      const int rows = (int)((M - tc.R0) < kTM ? (M - tc.R0) : kTM);
      const int cols = (int)((N - tc.C0) < kTN ? (N - tc.C0) : kTN);
      write_row_outputs(rstage, a.q_row, hN, tc, rows, cols, tid);
    }
    tile::write_col_outputs(cstage, sstage, a.q_col, a.s_col, M, N, tc, tid, a.sf_swz != 0);
    if (!more) break;
    w = wn;
  }
}

template <bool RHT_COL, bool NOCOPY = false>
cudaError_t launch_sr_rc(const QuantArgs& a, cudaStream_t s) {
  constexpr int kSmem = 2 * tile::kTileBytes + tile::kCStageBytes + tile::kSStageBytes + kRStageBytes + kRInvBytes +
                        256 * 4 + 2 * 8;
  auto kern = quant1d_sr_kernel<RHT_COL, NOCOPY>;
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kBlockThreads, kSmem, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTN - 1) / kTN);
  int64_t g = ntiles < cap ? ntiles : cap;
  if (g < 1) g = 1;
  CUtensorMap xmap;
  const cudaError_t me = make_tile_map(&xmap, a.x, a.M, a.N, a.ld);
  if (me != cudaSuccess) return me;
  kern<<<dim3((unsigned)g, 1, 1), kBlockThreads, kSmem, s>>>(a, xmap);
  return cudaGetLastError();
}

}  // namespace q1d
}  // namespace nvfp4
