// tile_pipeline.cuh -- shared-memory tile walk, staging and the cp.async
// tile loader.
//
// Persistent CTAs walk the tensor in 64 x 256 bf16 tiles (Walker).  The 1D
// quantize kernel fills its tiles with TMA (tma.cuh); the amax and 2D kernels
// use the loader here: while a tile is being processed the next one is
// already in flight as cp.async 16-byte global -> shared copies (zero-filled
// outside the tensor) into the other of two 32 KB buffers, completed by
// cp.async.wait_group plus __syncthreads.
//
// Loader tile layout: row r occupies 512 bytes; its 16-byte chunk c (eight
// bf16 values) sits at chunk c ^ ((c >> 3) & 1).  Reading a row's 32-byte
// block pair (chunks 2b, 2b+1) across 8 consecutive threads and reading one
// 4-byte column-pair word across a warp are then both bank-conflict free.
//
// Columnwise outputs go through a small staging area so that each column of
// the transposed copy receives its 32 code bytes (64 rows) in one store:
//   cstage: [4 row blocks][256 columns] x 8 code bytes   (8 KB)
//   sstage: [256 columns] x 4 scale bytes                (1 KB)
#pragma once

#include <cstdint>

namespace nvfp4 {
namespace tile {

constexpr int kTM = 64;
constexpr int kTN = 256;
constexpr int kRowBytes = kTN * 2;
constexpr int kTileBytes = kTM * kRowBytes;  // 32 KB
constexpr int kChunks = kTM * kTN / 8;       // 2048 chunks of 16 bytes
constexpr int kCStageBytes = 4 * kTN * 8;    // 8 KB
constexpr int kSStageBytes = kTN * 4;        // 1 KB

__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 3) & 1); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

struct Coord {
  int64_t R0, C0;
};

// Tile walk of a persistent CTA: tiles t = blockIdx.x + k*gridDim.x in
// row-major tile order (ntx tiles per row of tiles), with the (row, column)
// tile coordinates advanced incrementally instead of divided per tile.
// TN: tile width in columns (the 1D kernels without stochastic rounding walk
// 64 x 128 tiles).
template <int TN = kTN>
struct WalkerT {
  int64_t ty, tx;        // current tile
  int64_t step_y, step_x; // gridDim.x = step_y * ntx + step_x
  int64_t ntx, nty;
  __device__ __forceinline__ void init(int64_t M, int64_t N) {
    ntx = (N + TN - 1) / TN;
    nty = (M + kTM - 1) / kTM;
    if (ntx < 1) ntx = 1;
    ty = blockIdx.x / ntx;
    tx = blockIdx.x - ty * ntx;
    step_y = gridDim.x / ntx;
    step_x = gridDim.x - step_y * ntx;
  }
  __device__ __forceinline__ bool valid() const { return ty < nty; }
  __device__ __forceinline__ Coord coord() const { return {ty * kTM, tx * TN}; }
  __device__ __forceinline__ WalkerT next() const {
    WalkerT w = *this;
    w.tx += step_x;
    w.ty += step_y;
    if (w.tx >= ntx) {
      w.tx -= ntx;
      w.ty += 1;
    }
    return w;
  }
};
using Walker = WalkerT<>;

// Issue the async copies of one tile (NT threads, thread `tid`).
template <int NT>
__device__ __forceinline__ void load_async(uint8_t* buf, const uint16_t* x, int64_t M, int64_t N, int64_t ld,
                                           Coord tc, int tid) {
#pragma unroll
  for (int k = 0; k < kChunks / NT; ++k) {
    const int id = tid + k * NT;
    const int r = id >> 5, c = id & 31;
    const int64_t grow = tc.R0 + r, gcol = tc.C0 + 8 * c;
    const bool ok = grow < M && gcol < N;
    const uint16_t* src = ok ? x + grow * ld + gcol : x;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(buf + r * kRowBytes + swz(c) * 16)),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
  }
}

__device__ __forceinline__ void commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void wait_all_but_one() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Two 16-byte chunks (16 bf16 values) of row r starting at tile column 16*b.
__device__ __forceinline__ void read_row_block(const uint8_t* buf, int r, int b, uint32_t* wd) {
  const uint4 lo = *reinterpret_cast<const uint4*>(buf + r * kRowBytes + swz(2 * b) * 16);
  const uint4 hi = *reinterpret_cast<const uint4*>(buf + r * kRowBytes + swz(2 * b + 1) * 16);
  wd[0] = lo.x; wd[1] = lo.y; wd[2] = lo.z; wd[3] = lo.w;
  wd[4] = hi.x; wd[5] = hi.y; wd[6] = hi.z; wd[7] = hi.w;
}

// bf16x2 word holding tile columns (2p, 2p+1) of row r.
__device__ __forceinline__ uint32_t read_pair_word(const uint8_t* buf, int r, int p) {
  return *reinterpret_cast<const uint32_t*>(buf + r * kRowBytes + swz(p >> 2) * 16 + (p & 3) * 4);
}

// Stage the columnwise codes/scales of tile columns (2p, 2p+1), row block rb.
__device__ __forceinline__ void stage_col_pair(uint8_t* cstage, uint8_t* sstage, int p, int rb, uint2 c0, uint2 c1,
                                               uint32_t e0, uint32_t e1) {
  *reinterpret_cast<uint4*>(cstage + rb * (kTN * 8) + p * 16) = make_uint4(c0.x, c0.y, c1.x, c1.y);
  sstage[(2 * p) * 4 + rb] = (uint8_t)e0;
  sstage[(2 * p + 1) * 4 + rb] = (uint8_t)e1;
}

__device__ __forceinline__ void st_v8(uint8_t* p, uint2 a, uint2 b, uint2 c, uint2 d) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(p), "r"(a.x), "r"(a.y), "r"(b.x),
               "r"(b.y), "r"(c.x), "r"(c.y), "r"(d.x), "r"(d.y)
               : "memory");
}

// Byte offset of scale (r, c) in the tiled layout of block-scaled MMA
// operands: 128 x 4 tiles of 512 bytes in row-major tile order (ctiles tiles
// per tile row), (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4 inside a tile.
__device__ __forceinline__ int64_t sf_swz_off(int64_t r, int64_t c, int64_t ctiles) {
  return ((r >> 7) * ctiles + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// Padded staging (PAD = true) for writers whose lanes hold columns 8 apart:
// 16 bytes after every 16 columns of codes and 4 bytes after every 8 columns
// of scales spread such lanes over all banks.
constexpr int kCStageRowPad = kTN * 8 + (kTN / 16) * 16;          // 2304 bytes per row block
constexpr int kCStagePadBytes = 4 * kCStageRowPad;                // 9 KB
constexpr int kSStagePadBytes = kTN * 4 + (kTN / 8) * 4;          // 1152 bytes
__device__ __forceinline__ int cstage_off_pad(int rb, int c) { return rb * kCStageRowPad + 8 * c + 16 * (c >> 4); }
__device__ __forceinline__ int sstage_off_pad(int c) { return 4 * c + 4 * (c >> 3); }

// Write the staged columnwise outputs of one tile: tile column `c` (one per
// thread) gets its codes for up to 64 rows (32 bytes) and up to 4 scales.
// With swz the scales go to the tiled layout (their four row blocks stay
// four consecutive bytes there, as the tile origin is a multiple of 64 rows).
template <bool PAD = false>
__device__ __forceinline__ void write_col_outputs(const uint8_t* cstage, const uint8_t* sstage, uint8_t* q_col,
                                                  uint8_t* s_col, int64_t M, int64_t N, Coord tc, int c,
                                                  bool swz = false) {
  const int64_t gc = tc.C0 + c;
  if (gc >= N) return;
  int64_t nrb = (M - tc.R0) / 16;
  if (nrb > 4) nrb = 4;
  uint2 w[4];
#pragma unroll
  for (int rb = 0; rb < 4; ++rb)
    w[rb] = *reinterpret_cast<const uint2*>(cstage + (PAD ? cstage_off_pad(rb, c) : rb * (kTN * 8) + c * 8));
  uint8_t* dst = q_col + gc * (M / 2) + tc.R0 / 2;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(dst);
  if (nrb == 4 && (addr & 31) == 0) {
    st_v8(dst, w[0], w[1], w[2], w[3]);
  } else if (nrb == 4 && (addr & 15) == 0) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0].x, w[0].y, w[1].x, w[1].y);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[2].x, w[2].y, w[3].x, w[3].y);
  } else {
    for (int rb = 0; rb < nrb; ++rb) *reinterpret_cast<uint2*>(dst + 8 * rb) = w[rb];
  }
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(sstage + (PAD ? sstage_off_pad(c) : c * 4));
  uint8_t* sdst = s_col + (swz ? sf_swz_off(gc, tc.R0 / 16, (M / 16 + 3) / 4) : gc * (M / 16) + tc.R0 / 16);
  if (nrb == 4 && (reinterpret_cast<uintptr_t>(sdst) & 3) == 0) {
    *reinterpret_cast<uint32_t*>(sdst) = sw;
  } else {
    for (int rb = 0; rb < nrb; ++rb) sdst[rb] = (uint8_t)(sw >> (8 * rb));
  }
}

}  // namespace tile
}  // namespace nvfp4
