// gemm_kernel.cuh -- NVFP4 block-scaled GEMM on the fifth-generation tensor cores
// (the kernel; gemm.cu instantiates and launches it).
//
// D = alpha_a * alpha_b * (A * B^T), fp32 or bf16 out: A (M x K) and B (N x K)
// are NVFP4 operands exactly as nvfp4_quantize writes them with
// NVFP4_SF_SWIZZLED -- packed E2M1 codes, K contiguous (a rowwise copy, or a
// columnwise copy for a transposed operand), and E4M3 scales per 16 values
// along K in the tiled 128 x 4 layout -- so the quantizer's outputs feed the
// tensor cores without a re-layout ("NVFP4 revolutionizes AI training"
// headline page: Blackwell multiplies FP4 matrices natively).
//
// Persistent CTAs (one per SM) walk the 128 x 128 output tiles in groups of
// eight M tiles (see tile_coords), so that the CTAs in flight share A and B
// tiles in L2.  Six warps:
//   - warp 0 allocates 512 TMEM columns; its lane 0 is the producer: per
//     K step of 256 values it loads a 128 x 128-byte tile of A and of B with
//     TMA (128-byte swizzle, the K-major layout the MMA reads) and the two
//     2 KB scale blocks with bulk copies, into one of six shared-memory
//     stages, completion on the stage's "full" mbarrier;
//   - warps 6-9 (one TMEM lane quarter each) move each stage's scale blocks
//     from shared memory to TMEM (tcgen05.st; 16 bytes per lane = the 4 scale
//     bytes of rows l, l+32, l+64, l+96, in every lane quarter), off the MMA
//     warp's in-order path, and signal the stage's "scales" mbarrier;
//   - warp 1 lane 0 issues, per stage, four tcgen05.mma (kind::mxf4nvf4,
//     M = 128, N = 128, K = 64) into one of two fp32 accumulators in TMEM
//     (columns 0-127, 128-255), then a commit that frees the stage; after a
//     tile's last K step a commit hands the accumulator to the epilogue;
//   - warps 2-5 (one TMEM lane quarter each) read an accumulator, release it
//     to the MMA warp, apply alpha_a * alpha_b and store D, while the MMA warp
//     fills the other accumulator.
// Every wait is bounded (about a second); a wait that runs out writes
// NVFP4_ERR_PIPELINE to the status word, the loops stop, the tensor-core work
// already issued is drained, and TMEM is released on every path.
#pragma once

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace nvfp4 {
namespace gemmk {

constexpr int kBM = 128;
constexpr int kBK = 256;                         // FP4 values per K step (128 bytes of codes per row)
constexpr int kTileA = kBM * kBK / 2;            // 16 KB
constexpr int kSfBlock = 512;                    // scales of 128 rows x 64 values
constexpr int kSfBytes = (kBK / 64) * kSfBlock;  // 2 KB per 128 rows and stage
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 320;
constexpr int kSfWarp0 = 6;  // warps 6-9 move the scale blocks to TMEM

// Tile shapes: 128 x 128 output tiles with two accumulators (the epilogue of
// one tile overlaps the next tile's MMAs) and six stages, or 128 x 256 tiles
// with one accumulator and four stages -- a quarter fewer operand bytes per
// FLOP through shared memory, for an epilogue that the next tile's MMAs wait
// for until it has read the accumulator out (its stores overlap them only
// after the last chunk).  TMEM: accumulators in columns 0-255,
// per-stage scale factors from column 256 (A: 4 columns per MMA; B: 4 per
// 128 rows per MMA).
template <int BN>
struct Cfg {
  static constexpr int kBN = BN;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kAcc = BN == 256 ? 1 : 2;
  static constexpr int kTileB = BN * kBK / 2;              // 16 / 32 KB
  static constexpr int kSfbBytes = (BN / 128) * kSfBytes;  // 2 / 4 KB
  static constexpr int kStageBytes = kTileA + kTileB + kSfBytes + kSfbBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* barriers, TMEM address */ + 1024 /* alignment */;
  static constexpr uint32_t kSfCol0 = kAcc * BN;           // 256
  static constexpr uint32_t kSfbCols = 4 * (BN / 128);     // per MMA
  static constexpr uint32_t kSfStageCols = 16 + 4 * kSfbCols;
  static_assert(kSfCol0 + kStages * kSfStageCols <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Tile t -> (M tile, N tile), grouped: kGroupM consecutive M tiles are walked
// N tile by N tile, so the CTAs in flight cover a block of about kGroupM x
// (SMs / kGroupM) tiles and each A and B tile is shared by several of them.
#ifndef NVFP4_GEMM_GROUP_M
#define NVFP4_GEMM_GROUP_M 8
#endif
constexpr int64_t kGroupM = NVFP4_GEMM_GROUP_M;

__device__ __forceinline__ void tile_coords(int64_t t, int64_t tiles_m, int64_t tiles_n, int64_t& tm, int64_t& tn) {
  const int64_t per_group = kGroupM * tiles_n;
  const int64_t g = t / per_group, r = t - g * per_group;
  const int64_t m0 = g * kGroupM;
  const int64_t gm = (tiles_m - m0) < kGroupM ? (tiles_m - m0) : kGroupM;  // M tiles in this (last) group
  tm = m0 + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// NOCOPY (a test instantiation only): the producer arms the stage barriers
// but issues no copy, so every wait downstream runs out.
template <int BN, bool NOCOPY = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap) {
  using C = Cfg<BN>;
  constexpr int kStages = C::kStages, kStageBytes = C::kStageBytes, kTileB = C::kTileB, kAcc = C::kAcc;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
  const uint32_t accf0 = smem_u32(bars + 2 * kStages), acce0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  int* abort_flag = reinterpret_cast<int*>(bars + 2 * kStages + 6);
  const uint32_t sfr0 = smem_u32(bars + 2 * kStages + 7);  // per stage: scales in TMEM

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = (int)(a.K / kBK);
  const int64_t tiles_n = a.N / BN, tiles_m = a.M / kBM, tiles = tiles_m * tiles_n;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tma::mbar_init(full0 + 8 * s, 1);
      tma::mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tma::mbar_init(accf0 + 8 * b, 1);
      tma::mbar_init(acce0 + 8 * b, 4);  // one arrival per epilogue warp
    }
    tma::mbar_init(drain, 1);
    for (int st = 0; st < kStages; ++st) tma::mbar_init(sfr0 + 8 * st, 4);  // one arrival per scale warp
    *abort_flag = 0;
    tma::fence_barrier_init();
  }
  if (warp == 0) {
    tc5::alloc(smem_u32(tmem_slot), kTmemCols);
    tc5::relinquish_alloc_permit();
  }
  tc5::fence_before_thread_sync();
  __syncthreads();
  tc5::fence_after_thread_sync();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_v = abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // producer: TMA tiles of A and B, bulk copies of their scale blocks
      const int64_t sf_tiles_k = a.K / 64;  // 512-byte scale blocks per 128-row band
      int64_t g = 0;                        // K steps issued by this CTA
      for (int64_t t = blockIdx.x; t < tiles && !*abort_v; t += gridDim.x) {
        int64_t tm, tn;
        tile_coords(t, tiles_m, tiles_n, tm, tn);
        const uint8_t* sfa = a.sfa + tm * sf_tiles_k * kSfBlock;
        const uint8_t* sfb = a.sfb + tn * (BN / 128) * sf_tiles_k * kSfBlock;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = (int)(g % kStages);
          const uint32_t ph = (uint32_t)(g / kStages) & 1u;
          if (g >= kStages && !tma::wait(empty0 + 8 * s, ph ^ 1u)) {
            *abort_v = 1;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          const uint32_t full = full0 + 8 * s;
          tma::arrive_expect_tx(full, kStageBytes);
          if (NOCOPY) continue;
          tma::load_2d(smem_u32(st), &amap, kb * (kBK / 2), (int)(tm * kBM), full);
          tma::load_2d(smem_u32(st + kTileA), &bmap, kb * (kBK / 2), (int)(tn * BN), full);
          tc5::bulk_g2s(smem_u32(st + kTileA + kTileB), sfa + (int64_t)kb * kSfBytes, kSfBytes, full);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)  // B's 128-row bands: their scale blocks one after the other
            tc5::bulk_g2s(smem_u32(st + kTileA + kTileB + kSfBytes + h * kSfBytes),
                          sfb + h * sf_tiles_k * kSfBlock + (int64_t)kb * kSfBytes, kSfBytes, full);
        }
      }
      // No copy may still be landing in shared memory when the CTA exits: the
      // last fill of every stage has completed (the MMA thread waited for it)
      // unless the pipeline stopped early, so wait for those fills (bounded).
      for (int64_t j = (g > kStages ? g - kStages : 0); j < g && !NOCOPY; ++j)
        tma::wait(full0 + 8 * (int)(j % kStages), (uint32_t)(j / kStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer
      constexpr uint32_t idesc = tc5::idesc_e2m1_e4m3(kBM, BN);
      int64_t g = 0;
      int li = 0;  // tiles of this CTA
      for (int64_t t = blockIdx.x; t < tiles && !*abort_v; t += gridDim.x, ++li) {
        const int ab = li % kAcc, use = li / kAcc;
        const uint32_t acc = tmem + (uint32_t)(ab * BN);
        // the epilogue has read this accumulator's previous tile out
        if (use >= 1 && !tma::wait(acce0 + 8 * ab, (uint32_t)((use - 1) & 1))) {
          *abort_v = 1;
          break;
        }
        tc5::fence_after_thread_sync();
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = (int)(g % kStages);
          const uint32_t ph = (uint32_t)(g / kStages) & 1u;
          // the tiles have arrived and the scale warps have put the stage's scales in TMEM
          if (!tma::wait(full0 + 8 * s, ph) || !tma::wait(sfr0 + 8 * s, ph)) {
            *abort_v = 1;
            break;
          }
          tc5::fence_after_thread_sync();
          const uint8_t* st = smem + s * kStageBytes;
          const uint32_t a_base = smem_u32(st), b_base = smem_u32(st + kTileA);
          const uint32_t sf_base = tmem + C::kSfCol0 + (uint32_t)(s * C::kSfStageCols);
#pragma unroll
          for (int j = 0; j < kBK / 64; ++j) {
            const uint32_t sfa_t = sf_base + (uint32_t)(4 * j);
            const uint32_t sfb_t = sf_base + 16u + C::kSfbCols * (uint32_t)j;
            // K step j: 64 values = 32 bytes into each 128-byte swizzled row
            const uint64_t adesc = tc5::smem_desc(a_base + 32 * j, 16, 1024, tc5::kLayoutSwizzle128B);
            const uint64_t bdesc = tc5::smem_desc(b_base + 32 * j, 16, 1024, tc5::kLayoutSwizzle128B);
            tc5::mma_nvf4(acc, adesc, bdesc, idesc, sfa_t, sfb_t, kb > 0 || j > 0);
          }
          tc5::commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
        }
        if (*abort_v) break;
        tc5::commit(accf0 + 8 * ab);  // the accumulator is complete once these MMAs are
      }
      tc5::commit(drain);  // arrives when every MMA issued above has completed
    }
  } else if (warp >= kSfWarp0) {
    // scale warps: warp w writes TMEM lane quarter w % 4; every quarter gets the
    // same 16 bytes per lane (the four row groups of a 128 x 4 scale tile)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int64_t g = 0;
    bool stop = false;  // warp-uniform: every lane takes the same path to the .sync.aligned stores
    for (int64_t t = blockIdx.x; t < tiles && !stop; t += gridDim.x) {
      stop = __any_sync(0xFFFFFFFFu, *abort_v != 0);
      for (int kb = 0; kb < nk && !stop; ++kb, ++g) {
        const int s = (int)(g % kStages);
        const uint32_t ph = (uint32_t)(g / kStages) & 1u;
        const bool arrived = tma::wait(full0 + 8 * s, ph);
        if (!__all_sync(0xFFFFFFFFu, arrived)) {
          if (lane == 0) *abort_v = 1;
          stop = true;
          break;
        }
        const uint8_t* sf = smem + s * kStageBytes + kTileA + kTileB;
        const uint32_t sf_base = tmem + lane_base + C::kSfCol0 + (uint32_t)(s * C::kSfStageCols);
#pragma unroll
        for (int j = 0; j < kBK / 64; ++j) {
          const uint4 va = *reinterpret_cast<const uint4*>(sf + j * kSfBlock + 16 * lane);
          tc5::st_32x32b_x4(sf_base + (uint32_t)(4 * j), va);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            const uint4 vb = *reinterpret_cast<const uint4*>(sf + kSfBytes + h * kSfBytes + j * kSfBlock + 16 * lane);
            tc5::st_32x32b_x4(sf_base + 16u + C::kSfbCols * (uint32_t)j + 4u * h, vb);
          }
        }
        tc5::wait_st();
        tc5::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sfr0 + 8 * s) : "memory");
      }
    }
  } else {
    // epilogue: warp w reads TMEM lane quarter w % 4 = rows 32 * (w % 4) + lane of the tile
    const int q = warp & 3;
    const float scale = __fmul_rn(a.alpha_a[0], a.alpha_b[0]);
    int li = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++li) {
      const int ab = li % kAcc, use = li / kAcc;
      const bool ready = tma::wait(accf0 + 8 * ab, (uint32_t)(use & 1));
      // warp-uniform decision before the .sync.aligned TMEM loads
      if (!__all_sync(0xFFFFFFFFu, ready) || __any_sync(0xFFFFFFFFu, *abort_v != 0)) {
        if (lane == 0) *abort_v = 1;
        break;
      }
      tc5::fence_after_thread_sync();
      int64_t tm, tn;
      tile_coords(t, tiles_m, tiles_n, tm, tn);
      const int64_t row = tm * kBM + 32 * q + lane;
      const uint32_t acc = tmem + (uint32_t)(ab * BN) + ((uint32_t)(32 * q) << 16);
      auto release = [&]() {  // the accumulator is in registers: hand it back to the MMA warp
        tc5::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acce0 + 8 * ab) : "memory");
      };
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc5::ld_32x32b_x32(acc + (uint32_t)(32 * c), r);
        tc5::wait_ld();
        if (c == BN / 32 - 1) release();
        const int64_t col = tn * BN + 32 * c;
        if (a.out_bf16) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.d) + row * a.ldd + col;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * v + 0]), scale), __fmul_rn(__uint_as_float(r[8 * v + 1]), scale));
            w.y = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * v + 2]), scale), __fmul_rn(__uint_as_float(r[8 * v + 3]), scale));
            w.z = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * v + 4]), scale), __fmul_rn(__uint_as_float(r[8 * v + 5]), scale));
            w.w = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * v + 6]), scale), __fmul_rn(__uint_as_float(r[8 * v + 7]), scale));
            *reinterpret_cast<uint4*>(dst + 8 * v) = w;
          }
        } else {
          float* dst = reinterpret_cast<float*>(a.d) + row * a.ldd + col;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 f;
            f.x = __fmul_rn(__uint_as_float(r[4 * v + 0]), scale);
            f.y = __fmul_rn(__uint_as_float(r[4 * v + 1]), scale);
            f.z = __fmul_rn(__uint_as_float(r[4 * v + 2]), scale);
            f.w = __fmul_rn(__uint_as_float(r[4 * v + 3]), scale);
            *reinterpret_cast<float4*>(dst + 4 * v) = f;
          }
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();
  // drain the tensor-core work issued by the MMA thread (its last commit), then free TMEM
  const bool drained = tma::wait(drain, 0);
  if (tid == 0 && (*abort_v || !drained) && a.status) atomicExch(a.status, kStatusPipeline);
  tc5::fence_before_thread_sync();
  __syncthreads();
  if (warp == 0) tc5::dealloc(tmem, kTmemCols);
}

template <int BN, bool NOCOPY = false>
cudaError_t launch(const GemmArgs& a, cudaStream_t s) {
  using C = Cfg<BN>;
  auto kern = gemm_nvf4_kernel<BN, NOCOPY>;
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kThreads, C::kSmemBytes, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  CUtensorMap amap, bmap;
  cudaError_t e = make_codes_map(&amap, a.qa, a.M, a.K / 2, kBK / 2, kBM);
  if (e != cudaSuccess) return e;
  e = make_codes_map(&bmap, a.qb, a.N, a.K / 2, kBK / 2, BN);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.M / kBM) * (a.N / BN);
  const int64_t grid = tiles < cap ? tiles : cap;
  kern<<<(unsigned)grid, kThreads, C::kSmemBytes, s>>>(a, amap, bmap);
  return cudaGetLastError();
}

}  // namespace gemmk
}  // namespace nvfp4
