#pragma once
// quant1d_kernel.cuh -- fused rowwise + columnwise NVFP4 quantization with 1x16 blocks.
//
// One read of X produces both copies.  Persistent CTAs stream 64 x 256 bf16
// tiles into double-buffered shared memory with TMA bulk tensor copies (four
// 64 x 64 boxes per tile, 128-byte swizzle, completion on an mbarrier; one
// thread issues them while the CTA works on the other buffer), then
//   - the rowwise pass gives each thread whole 16-column blocks (two 128-bit
//     shared loads) and stores their codes directly (32 bytes per row), and
//   - the columnwise pass gives each thread a column pair over 16 rows (sixteen
//     32-bit shared loads, one bf16x2 word per row) and stages the codes, so
//     that each column of the transposed copy is written as one 32-byte store,
// so every block's scale, rounding and 4/6 choice happen in one thread's
// registers.  Element arithmetic uses packed f32x2 operations, which halve
// the issue slots of the multiplies and fused multiply-adds.  The per-block
// code is straight-line: scale bytes come from a division-free quotient (see
// quotient_rn), the RHT flags and the 4/6 rule are template parameters.
//
// With stochastic rounding on both copies, one Philox4x32-10 call per element
// serves both.  Without 4/6 and without a rowwise Hadamard transform that
// case runs in quant1d_sr_kernel.cuh (both roundings in the columnwise pass);
// here, for 4/6 or a rowwise transform, the rowwise pass uses word 0 and
// parks word 1 in shared memory for the columnwise pass (that 64 KB stash
// leaves room for one tile buffer, so those kernels load each tile after the
// previous one is done and rely on their second CTA per SM for overlap).
//
// Sources: "Four Over Six (4/6)" technical summary (Problem statement,
// Methodology, Implementation details) and "Pretraining Large Language Models
// with NVFP4" sections 1, 2b and 2d.
#include "quant1d_common.cuh"

#ifndef NVFP4_Q1D_MIN_CTAS
#define NVFP4_Q1D_MIN_CTAS 3  // resident CTAs per SM the register budget is sized for
#endif

namespace nvfp4 {
namespace q1d {

constexpr int kStashBytes = kTM * kTN * 4;  // Philox word 1 per element, 64 KB
// Tile width (columns) of the 1D kernel: 64 x 128 tiles for plain
// round-to-nearest, whose CTAs are bound by the latency of a tile's work (a
// narrower tile halves it, and with it the cost of the launch's first and
// last rounds of tiles: RN R+C 32.6 -> 30.7 us on 8192 x 5120); 64 x 256
// with 4/6, RHT or SR (the narrow tile measured 1-9 % slower there, and the
// SR stash is laid out for 256 columns).
template <bool Q46, bool SR, int RHT>
constexpr int tile_width() { return (Q46 || SR || RHT != 0) ? kTN : kTN / 2; }

// Byte offset of the stash word of tile row r, tile column c.  A row is
// 1 KB (256 words); its 16-byte chunk q = c / 4 sits at
// q ^ ((q >> 3) & 7) ^ ((r & 1) << 1), so that the rowwise pass's 16-byte
// stores from a quarter warp (two rows, four blocks) fall in eight distinct
// bank groups.
__device__ __forceinline__ uint32_t stash_off(int r, int c) {
  const int q = c >> 2;
  return (uint32_t)r * 1024u + (uint32_t)((q ^ ((q >> 3) & 7) ^ ((r & 1) << 1)) << 4) + (uint32_t)(c & 3) * 4u;
}

// v = z * inv for 16 values (packed), then SR rounding or, for a max-4
// candidate with a subnormal scale byte, the clamp to +-4 that RN needs.
template <bool SR>
__device__ __forceinline__ void scale16(const float* z, float inv, uint32_t e, float Q, const uint32_t* w, float* v) {
  const float2 inv2 = make_float2(inv, inv);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 r = mul2(make_float2(z[2 * j], z[2 * j + 1]), inv2);
    v[2 * j] = r.x;
    v[2 * j + 1] = r.y;
  }
  if (SR) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = sr_round(v[j], Q, w[j]);
  } else if (Q == 4.0f && max4_needs_clamp(e)) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = fminf(fmaxf(v[j], -4.0f), 4.0f);
  }
}

// Codes of one 4/6 candidate and its score, computed pair by pair so that
// only the code bytes and eight partial sums stay live: for each pair the
// scaled values are encoded, the codes decoded back to grid values, and
// err = z - val*d (rounded once) folded into the first level of the tree.
// MAE sums |err|, MSE sums err*err, both over the perfect binary tree in
// block order; MAXERR takes max |err|.
template <bool SR, int SEL>
__device__ __forceinline__ float candidate16(const float* z, uint32_t e, float2 di, float Q, const uint32_t* w,
                                             uint2& codes) {
  const float2 inv2 = make_float2(di.y, di.y);
  const float2 nd = make_float2(-di.x, -di.x);
  const bool clamp = !SR && Q == 4.0f && max4_needs_clamp(e);
  float t[8];
  uint32_t cw[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 r = mul2(make_float2(z[8 * half + 2 * j], z[8 * half + 2 * j + 1]), inv2);
      v[2 * j] = r.x;
      v[2 * j + 1] = r.y;
    }
    if (SR) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = sr_round(v[j], Q, w[8 * half + j]);
    } else if (clamp) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = fminf(fmaxf(v[j], -4.0f), 4.0f);
    }
    uint32_t h2[4];
    cw[half] = e2m1x8_enc_dec(v, h2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 zz = make_float2(z[8 * half + 2 * j], z[8 * half + 2 * j + 1]);
      const float2 err = fma2(f16x2_to_f32x2(h2[j]), nd, zz);  // z - val*d, rounded once
      float tj;
      if (SEL == kSelMSE) {
        const float2 sq = mul2(err, err);
        tj = __fadd_rn(sq.x, sq.y);
      } else if (SEL == kSelMax) {
        tj = fmaxf(fabsf(err.x), fabsf(err.y));
      } else {
        tj = __fadd_rn(fabsf(err.x), fabsf(err.y));
      }
      t[4 * half + j] = tj;
    }
  }
  codes = make_uint2(cw[0], cw[1]);
  if (SEL == kSelMax)
    return fmaxf(fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])), fmaxf(fmaxf(t[4], t[5]), fmaxf(t[6], t[7])));
  // ((t0+t1)+(t2+t3)) + ((t4+t5)+(t6+t7)), two sums per packed add
  const float2 a = add2(make_float2(t[0], t[4]), make_float2(t[1], t[5]));
  const float2 b = add2(make_float2(t[2], t[6]), make_float2(t[3], t[7]));
  const float2 c = add2(a, b);
  return __fadd_rn(c.x, c.y);
}

// One block at the given scale bytes: the standard max-6 candidate and, with
// 4/6, the max-4 candidate; the max-4 one is kept only if its score is
// strictly lower.
template <bool Q46, bool SR, int SEL>
__device__ __forceinline__ void quant_block16(const float* z, const CopyScales& sc, const uint32_t* w, uint32_t e6,
                                              uint32_t e4, uint2& codes, uint32_t& e) {
  const float2 di6 = sc.tbl[e6];
  if (!Q46) {
    float v[16];
    scale16<SR>(z, di6.y, e6, 6.0f, w, v);
    codes = make_uint2(e2m1x8(v), e2m1x8(v + 8));
    e = e6;
    return;
  }
  uint2 c6, c4;
  const float s6 = candidate16<SR, SEL>(z, e6, di6, 6.0f, w, c6);
  const float s4 = candidate16<SR, SEL>(z, e4, sc.tbl[e4], 4.0f, w, c4);
  const bool four = s4 < s6;
  codes = four ? c4 : c6;
  e = four ? e4 : e6;
}

// Scale bytes of a block with maximum b (e4 only with 4/6).
template <bool Q46>
__device__ __forceinline__ void block_bytes(float b, const CopyScales& sc, uint32_t& e6, uint32_t& e4) {
  e6 = scale_byte(b, sc.den6, sc.rden6);
  e4 = Q46 ? scale_byte(b, sc.den4, sc.rden4) : 0u;
}

// RHT bit 0: Hadamard on the rowwise copy; bit 1: on the columnwise copy.
// NOCOPY (a test instantiation only): arm the tile barriers but issue no copy.
template <bool ROW, bool COL, bool Q46, bool SR, int SEL, int RHT, bool NOCOPY = false>
__global__ void __launch_bounds__(kBlockThreads, SR ? 2 : NVFP4_Q1D_MIN_CTAS)
    quant1d_kernel(const QuantArgs a, const __grid_constant__ CUtensorMap xmap) {
  constexpr bool kRhtRow = (RHT & 1) != 0, kRhtCol = (RHT & 2) != 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr bool kStash = SR && ROW && COL;
  // With the 64 KB stash a second tile buffer would leave room for one CTA
  // per SM; a single buffer fits two, whose loads overlap each other's math.
  constexpr bool kDB = !kStash;
  constexpr int kBufs = kDB ? 2 : 1;
  constexpr int kTW = tile_width<Q46, SR, RHT>(), kTileBytes = kTM * kTW * 2, kBoxes = kTW / 64;
  uint8_t* bufs = smem;                                      // 1 or 2 tiles (1024-aligned)
  uint8_t* cstage = smem + kBufs * kTileBytes;               // 8 KB
  uint8_t* sstage = cstage + tile::kCStageBytes;             // 1 KB
  float2* tbl = reinterpret_cast<float2*>(sstage + tile::kSStageBytes);  // 2 x 128 (d, 1/d)
  uint8_t* stash = reinterpret_cast<uint8_t*>(tbl + 256);    // 64 KB with kStash
  // Scale bytes never exceed 0x7E (448), so entry 127 of each table is free:
  // it holds the tile barrier of buffer 0 (R table) and buffer 1 (C table).
  const uint32_t bar0 = tile::smem_u32(tbl + 127), bar1 = tile::smem_u32(tbl + 255);

  // a2: alpha = amax / (6*448), or amax / (6*256) with 4/6
  float alpha_r, alpha_c;
  if (!begin_tensor(a, ROW, COL, Q46 ? kAlphaDen46 : kAlphaDen, smem, alpha_r, alpha_c)) return;

  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x;
  auto issue = [&](int b, const tile::Coord& c) {
    const uint32_t bar = b ? bar1 : bar0;
    tma::arrive_expect_tx(bar, kTileBytes);
    if (NOCOPY) return;
    const uint32_t dst = tile::smem_u32(bufs + b * kTileBytes);
#pragma unroll
    for (int j = 0; j < kBoxes; ++j) tma::load_2d(dst + j * 8192, &xmap, (int)c.C0 + 64 * j, (int)c.R0, bar);
  };
  tile::WalkerT<kTW> w;
  w.init(M, N);
  if (tid == 0) {
    tma::mbar_init(bar0, 1);
    tma::mbar_init(bar1, 1);
    tma::fence_barrier_init();
    if (w.valid()) issue(0, w.coord());  // the first tile is in flight while the tables are built
  }
  if ((tid & 127) != 127) tbl[tid] = scale_entry(tid & 127, (tid >> 7) ? alpha_c : alpha_r);
  __syncthreads();  // barriers and tables ready
  const CopyScales scR = make_scales(alpha_r, tbl);
  const CopyScales scC = make_scales(alpha_c, tbl + 128);
  const uint32_t signs = (kRhtRow || kRhtCol) ? rht_sign_bits(a.rht_k0, a.rht_k1) : 0u;

  // Shared tile = kTW / 64 boxes of 64 columns as the TMA writes them: box j
  // at 8 KB * j, row r at 128 * r, 16-byte chunk c at (c ^ (r & 7)) * 16.
  // Fixed per-thread roles (relative to a tile's origin):
  //  rowwise    tile row rr = 8*warp + lane/4, blocks rq + 4k (k < kTW/64):
  //             block rq + 4k is chunks 2rq, 2rq+1 of box k, so a quarter
  //             warp (rows rr, rr+1; four blocks each) hits eight distinct
  //             bank groups, and each row's four code words are 32 bytes
  //  columnwise column pair cp_p, row blocks cp_rb0 + kRbStep * k: a warp
  //             reads one 128-byte box row per load
  const int lane = tid & 31;
  const int rr = 8 * (tid >> 5) + (lane >> 2), rq = lane & 3;
  const uint32_t r_chunk0 = rr * 128 + ((uint32_t)((2 * rq) ^ (lane >> 2)) << 4);  // second chunk: ^ 16
  const int64_t hN = N / 2, sN = N / 16;
  constexpr int kPairs = kTW / 2;                    // column pairs of a tile
  constexpr int kRbStep = kBlockThreads / kPairs;    // threads per column pair (row blocks apart)
  constexpr int kColTasks = 4 / kRbStep;             // row blocks per thread
  const int cp_p = tid % kPairs, cp_rb0 = tid / kPairs;
  const uint32_t c_base = (cp_p >> 5) * 8192 + (cp_p & 3) * 4;
  const uint32_t c_chunk = (uint32_t)((cp_p & 31) >> 2) << 4;

  for (int it = 0; w.valid(); w = w.next(), ++it) {
    const int b = kDB ? (it & 1) : 0;
    uint8_t* buf = bufs + b * kTileBytes;
    if (tid == 0) {
      if (kDB) {
        const tile::WalkerT<kTW> wn = w.next();
        if (wn.valid()) issue(b ^ 1, wn.coord());  // that buffer was released by the last barrier
      } else if (it > 0) {
        issue(0, w.coord());
      }
    }
    const uint32_t parity = kDB ? ((it >> 1) & 1) : (it & 1);
    const bool arrived = tma::wait(b ? bar1 : bar0, parity);
    if (!__syncthreads_and(arrived)) {
      // a copy did not arrive in time: report it, give the copies in flight
      // one more bounded wait, and stop
      if (tid == 0) {
        if (a.status) atomicExch(a.status, kStatusPipeline);
        tma::wait(b ? bar1 : bar0, parity);
        if (kDB && w.next().valid()) tma::wait(b ? bar0 : bar1, ((it + 1) >> 1) & 1);
      }
      return;
    }
    const tile::Coord tc = w.coord();
    const int64_t R0 = tc.R0, C0 = tc.C0;
    const int rows = (int)((M - R0) < kTM ? (M - R0) : kTM);
    const int cols = (int)((N - C0) < kTW ? (N - C0) : kTW);
    const bool cp_ok = 2 * cp_p < cols;

    // ---- rowwise copy: one 16-column block per task, kBoxes tasks per thread
    if (ROW && rr < rows) {
      uint8_t* qt = a.q_row + (R0 + rr) * hN + C0 / 2 + 8 * rq;
      // scale of block rq + 4k: plain layout st + 4k; tiled layout st + 512k
      uint8_t* st = a.s_row + (a.sf_swz ? tile::sf_swz_off(R0 + rr, C0 / 16 + rq, (sN + 3) / 4)
                                        : (R0 + rr) * sN + C0 / 16 + rq);
      const int st_step = a.sf_swz ? 512 : 4;
      const uint64_t ct = a.ctr_off + (uint64_t)((R0 + rr) * N + C0 + 16 * rq);
#pragma unroll
      for (int k = 0; k < kBoxes; ++k) {  // block rq + 4k of row rr
        if (16 * (rq + 4 * k) >= cols) break;
        uint32_t wd[8];
        {
          const uint4 lo = *reinterpret_cast<const uint4*>(buf + k * 8192 + r_chunk0);
          const uint4 hi = *reinterpret_cast<const uint4*>(buf + k * 8192 + (r_chunk0 ^ 16u));
          wd[0] = lo.x; wd[1] = lo.y; wd[2] = lo.z; wd[3] = lo.w;
          wd[4] = hi.x; wd[5] = hi.y; wd[6] = hi.z; wd[7] = hi.w;
        }
        if (kRhtRow) {
#pragma unroll
          for (int j = 0; j < 8; ++j) wd[j] ^= rht_mask_row(signs, j);  // s . z
        }
        float z[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = bf16x2_to_f32x2(wd[j]);
          z[2 * j] = f.x;
          z[2 * j + 1] = f.y;
        }
        float bmax;
        if (kRhtRow) {
          wht16(z);
          bmax = 0.0f;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float2 y = mul2(make_float2(z[j], z[j + 1]), make_float2(0.25f, 0.25f));
            z[j] = y.x;
            z[j + 1] = y.y;
            bmax = fmaxf(bmax, fmaxf(fabsf(y.x), fabsf(y.y)));
          }
        } else {
          bmax = block_absmax16(wd);
        }
        uint32_t e6, e4;
        block_bytes<Q46>(bmax, scR, e6, e4);
        uint32_t w[16];
        if (SR) {
          uint32_t w1[16];
          philox_group_w01<16, kStash>(ct + (uint64_t)(64 * k), 1u, a.sr_k0, a.sr_k1, w, w1);
          if (kStash) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(stash + stash_off(rr, 16 * (rq + 4 * k) + 4 * q)) =
                  make_uint4(w1[4 * q], w1[4 * q + 1], w1[4 * q + 2], w1[4 * q + 3]);
          }
        }
        uint2 codes;
        uint32_t e;
        quant_block16<Q46, SR, SEL>(z, scR, w, e6, e4, codes, e);
        *reinterpret_cast<uint2*>(qt + 32 * k) = codes;
        st[st_step * k] = (uint8_t)e;
      }
    }
    if (kStash) __syncthreads();

    // ---- columnwise copy: one column pair x 16 rows per task, kColTasks tasks per thread
    if (COL && cp_ok) {
      const int p = cp_p;
      // both tasks in flight at once, except with SR (its register budget is spent on Philox)
      constexpr int kColUnroll = SR ? 1 : 2;
#pragma unroll kColUnroll
      for (int k = 0; k < kColTasks; ++k) {  // row block rb of column pair p (both columns)
        const int rb = cp_rb0 + kRbStep * k;
        if (16 * rb >= rows) break;
        uint32_t wd[16];
        const uint8_t* cb = buf + c_base + rb * 2048;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wd[i] = *reinterpret_cast<const uint32_t*>(cb + i * 128 + (c_chunk ^ ((uint32_t)(i & 7) << 4)));
        // both columns' maxima at once (low half = column 2p, high half = 2p+1)
        uint32_t m2 = 0u;
        if (!kRhtCol) {
          uint32_t t8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t8[i] = absmax_bf16x2(wd[2 * i], wd[2 * i + 1]);
          m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(t8[0], t8[1]), absmax_bf16x2(t8[2], t8[3])),
                             absmax_bf16x2(absmax_bf16x2(t8[4], t8[5]), absmax_bf16x2(t8[6], t8[7]))) &
               0x7FFF7FFFu;
        }
        float zz[2][16];
        float bm[2] = {bf16_lo(m2), bf16_hi(m2)};
        if (kRhtCol) {  // both columns' 16-vectors at once, as pairs
          float2 zp[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) zp[i] = bf16x2_to_f32x2(wd[i] ^ rht_mask_col(signs, i));
          wht16_x2(zp);
          bm[0] = bm[1] = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 y = mul2(zp[i], make_float2(0.25f, 0.25f));
            zz[0][i] = y.x;
            zz[1][i] = y.y;
            bm[0] = fmaxf(bm[0], fabsf(y.x));
            bm[1] = fmaxf(bm[1], fabsf(y.y));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 f = bf16x2_to_f32x2(wd[i]);
            zz[0][i] = f.x;
            zz[1][i] = f.y;
          }
        }
        uint32_t e6[2], e4[2];
        block_bytes<Q46>(bm[0], scC, e6[0], e4[0]);
        block_bytes<Q46>(bm[1], scC, e6[1], e4[1]);
        uint2 codes[2];
        uint32_t es[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cc = 2 * p + h;  // tile column
          uint32_t w[16];
          if (SR) {
            if (kStash) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                w[i] = *reinterpret_cast<const uint32_t*>(stash + stash_off(16 * rb + i, cc));
            } else {
              uint32_t w0[16];
              philox_group_w01<16, true>(a.ctr_off + (uint64_t)((R0 + 16 * rb) * N + C0 + cc), (uint32_t)N, a.sr_k0,
                                 a.sr_k1, w0, w);
            }
          }
          quant_block16<Q46, SR, SEL>(zz[h], scC, w, e6[h], e4[h], codes[h], es[h]);
        }
        tile::stage_col_pair(cstage, sstage, p, rb, codes[0], codes[1], es[0], es[1]);
      }
    }
    __syncthreads();  // tile buffer free for the next copy; staging complete
    if (COL && tid < kTW) tile::write_col_outputs(cstage, sstage, a.q_col, a.s_col, M, N, tc, tid, a.sf_swz != 0);
  }
}

template <bool ROW, bool COL, bool Q46, bool SR, int SEL, int RHT, bool NOCOPY = false>
cudaError_t launch(const QuantArgs& a, cudaStream_t s) {
  constexpr bool kStash = SR && ROW && COL;
  constexpr int kTW = tile_width<Q46, SR, RHT>();
  constexpr int kSmem = (kStash ? 1 : 2) * (kTM * kTW * 2) + tile::kCStageBytes + tile::kSStageBytes + 256 * 8 +
                        (kStash ? kStashBytes : 0);
  auto kern = quant1d_kernel<ROW, COL, Q46, SR, SEL, RHT, NOCOPY>;
  // once per device: opt in to the dynamic shared memory and size the
  // persistent grid from the occupancy
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kBlockThreads, kSmem, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  // persistent grid: every resident CTA slot, or one CTA per tile if fewer
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTW - 1) / kTW);
  int64_t g = ntiles < cap ? ntiles : cap;
  if (g < 1) g = 1;
  CUtensorMap xmap;
  const cudaError_t me = make_tile_map(&xmap, a.x, a.M, a.N, a.ld);
  if (me != cudaSuccess) return me;
  const dim3 grid((unsigned)g, 1, 1);
  kern<<<grid, kBlockThreads, kSmem, s>>>(a, xmap);
  return cudaGetLastError();
}

// Stochastic rounding on both copies without 4/6 and without a rowwise
// Hadamard transform runs in quant1d_sr_kernel (launch_quant1d_sr_rc).
template <bool ROW, bool COL, bool Q46, int SEL, int RHT>
cudaError_t launch_sr(const QuantArgs& a, bool sr, cudaStream_t s) {
  if constexpr (ROW && COL && !Q46 && (RHT & 1) == 0) {
    return sr ? launch_quant1d_sr_rc(a, RHT == 2, s) : launch<ROW, COL, Q46, false, SEL, RHT>(a, s);
  } else {
    return sr ? launch<ROW, COL, Q46, true, SEL, RHT>(a, s) : launch<ROW, COL, Q46, false, SEL, RHT>(a, s);
  }
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
