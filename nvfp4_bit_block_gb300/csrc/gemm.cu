// gemm.cu -- NVFP4 block-scaled GEMM on the fifth-generation tensor cores.
//
// D = alpha_a * alpha_b * (A * B^T), fp32 out: A (M x K) and B (N x K) are
// NVFP4 operands exactly as nvfp4_quantize writes them with
// NVFP4_SF_SWIZZLED -- packed E2M1 codes, K contiguous (a rowwise copy, or a
// columnwise copy for a transposed operand), and E4M3 scales per 16 values
// along K in the tiled 128 x 4 layout -- so the quantizer's outputs feed the
// tensor cores without a re-layout ("NVFP4 revolutionizes AI training"
// headline page: Blackwell multiplies FP4 matrices natively).
//
// One CTA computes a 128 x 128 tile of D over all of K.  Four warps:
//   - warp 0 allocates 256 TMEM columns; its lane 0 is the producer: per
//     K step of 256 values it loads a 128 x 128-byte tile of A and of B with
//     TMA (128-byte swizzle, the K-major layout the MMA reads) and the two
//     2 KB scale blocks with bulk copies, into one of four shared-memory
//     stages, completion on the stage's "full" mbarrier;
//   - warp 1 lane 0 issues, per stage, four scale copies to TMEM and four
//     tcgen05.mma (kind::mxf4nvf4, M = 128, N = 128, K = 64, fp32 accumulator
//     in TMEM columns 0-127), then a commit that frees the stage;
//   - all four warps then read the accumulator (one TMEM lane quarter each),
//     apply alpha_a * alpha_b and store D.
// Every wait is bounded (about a second); a wait that runs out writes
// NVFP4_ERR_PIPELINE to the status word, and TMEM is released on every path.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace nvfp4 {
namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kBK = 256;                         // FP4 values per K step (128 bytes of codes per row)
constexpr int kStages = 4;
constexpr int kTileA = kBM * kBK / 2;            // 16 KB
constexpr int kTileB = kBN * kBK / 2;            // 16 KB
constexpr int kSfBlock = 512;                    // scales of 128 rows x 64 values
constexpr int kSfBytes = (kBK / 64) * kSfBlock;  // 2 KB per operand and stage
constexpr int kStageBytes = kTileA + kTileB + 2 * kSfBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* barriers, TMEM address */ + 1024 /* alignment */;
constexpr uint32_t kTmemCols = 256;              // accumulator 0-127, scale factors 128-255
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages), done = smem_u32(bars + 2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t m0 = (int64_t)blockIdx.y * kBM, n0 = (int64_t)blockIdx.x * kBN;
  const int nk = (int)(a.K / kBK);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tma::mbar_init(full0 + 8 * s, 1);
      tma::mbar_init(empty0 + 8 * s, 1);
    }
    tma::mbar_init(done, 1);
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

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // producer: TMA tiles of A and B, bulk copies of their scale blocks
    const int64_t sf_tiles_k = a.K / 64;  // 512-byte scale blocks per 128-row band
    const uint8_t* sfa = a.sfa + (blockIdx.y * sf_tiles_k) * kSfBlock;
    const uint8_t* sfb = a.sfb + (blockIdx.x * sf_tiles_k) * kSfBlock;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (uint32_t)(kb / kStages) & 1u;
      if (kb >= kStages && !tma::wait(empty0 + 8 * s, ph ^ 1u)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + s * kStageBytes;
      const uint32_t full = full0 + 8 * s;
      tma::arrive_expect_tx(full, kStageBytes);
      tma::load_2d(smem_u32(st), &amap, kb * (kBK / 2), (int)m0, full);
      tma::load_2d(smem_u32(st + kTileA), &bmap, kb * (kBK / 2), (int)n0, full);
      tc5::bulk_g2s(smem_u32(st + kTileA + kTileB), sfa + (int64_t)kb * kSfBytes, kSfBytes, full);
      tc5::bulk_g2s(smem_u32(st + kTileA + kTileB + kSfBytes), sfb + (int64_t)kb * kSfBytes, kSfBytes, full);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = tc5::idesc_e2m1_e4m3(kBM, kBN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (uint32_t)(kb / kStages) & 1u;
      if (!tma::wait(full0 + 8 * s, ph)) {
        ok = false;
        break;
      }
      tc5::fence_after_thread_sync();
      const uint8_t* st = smem + s * kStageBytes;
      const uint32_t a_base = smem_u32(st), b_base = smem_u32(st + kTileA);
      const uint32_t sfa_base = smem_u32(st + kTileA + kTileB), sfb_base = sfa_base + kSfBytes;
#pragma unroll
      for (int j = 0; j < kBK / 64; ++j) {
        const uint32_t sfa_t = tmem + 128u + (uint32_t)(s * 32 + 4 * j);
        const uint32_t sfb_t = tmem + 128u + (uint32_t)(s * 32 + 16 + 4 * j);
        tc5::cp_32x128b_warpx4(sfa_t, tc5::smem_desc(sfa_base + j * kSfBlock, 0, 128, tc5::kLayoutNone));
        tc5::cp_32x128b_warpx4(sfb_t, tc5::smem_desc(sfb_base + j * kSfBlock, 0, 128, tc5::kLayoutNone));
        // K step j: 64 values = 32 bytes into each 128-byte swizzled row
        const uint64_t adesc = tc5::smem_desc(a_base + 32 * j, 16, 1024, tc5::kLayoutSwizzle128B);
        const uint64_t bdesc = tc5::smem_desc(b_base + 32 * j, 16, 1024, tc5::kLayoutSwizzle128B);
        tc5::mma_nvf4(tmem, adesc, bdesc, idesc, sfa_t, sfb_t, kb > 0 || j > 0);
      }
      tc5::commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
    }
    tc5::commit(done);  // arrives when every MMA issued above has completed
  }
  __syncwarp();
  if (!ok && a.status) atomicExch(a.status, kStatusPipeline);

  // epilogue: lane quarter `warp` of the accumulator = rows m0 + 32*warp + lane
  const bool finished = tma::wait(done, 0);
  __syncwarp();
  tc5::fence_after_thread_sync();
  if (finished) {
    const float scale = __fmul_rn(a.alpha_a[0], a.alpha_b[0]);
    float* drow = a.d + (m0 + 32 * warp + lane) * a.ldd + n0;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      tc5::ld_32x32b_x32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(32 * c), r);
      tc5::wait_ld();
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v;
        v.x = __fmul_rn(__uint_as_float(r[4 * q + 0]), scale);
        v.y = __fmul_rn(__uint_as_float(r[4 * q + 1]), scale);
        v.z = __fmul_rn(__uint_as_float(r[4 * q + 2]), scale);
        v.w = __fmul_rn(__uint_as_float(r[4 * q + 3]), scale);
        *reinterpret_cast<float4*>(drow + 32 * c + 4 * q) = v;
      }
    }
  } else if (lane == 0 && a.status) {
    atomicExch(a.status, kStatusPipeline);
  }
  tc5::fence_before_thread_sync();
  __syncthreads();
  if (warp == 0) tc5::dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  static std::atomic<int> configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_relaxed);
  }
  CUtensorMap amap, bmap;
  e = make_codes_map(&amap, a.qa, a.M, a.K / 2, kBK / 2, kBM);
  if (e != cudaSuccess) return e;
  e = make_codes_map(&bmap, a.qb, a.N, a.K / 2, kBK / 2, kBN);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(a.N / kBN), (unsigned)(a.M / kBM), 1);
  gemm_nvf4_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, amap, bmap);
  return cudaGetLastError();
}

}  // namespace nvfp4
