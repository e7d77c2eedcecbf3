// amax.cu -- tensor amax for the rowwise and the columnwise copy.
//
// "Four Over Six (4/6)" technical summary, Implementation details: the global
// tensor scale comes from the tensor's largest magnitude.  A copy that is
// Hadamard-transformed ("Pretraining Large Language Models with NVFP4"
// section 2b) takes the largest magnitude of its transformed 16-vectors,
// computed with exactly the butterfly the quantize kernel uses, so the scale
// always covers the values that are quantized.
//
// Two kernels:
//   - amax_flat_kernel: a contiguous tensor without a transform is one flat
//     array; a persistent grid streams it with four 128-bit loads in flight per
//     thread and a NaN-propagating packed bf16 abs-max;
//   - amax_tile_kernel: a padded row stride or a transformed copy uses the
//     quantize kernels' persistent, double-buffered 64 x 256 shared-memory
//     tiles (tile_pipeline.cuh) and their two passes.
// Maxima are combined as the bit patterns of non-negative floats (unsigned
// order equals float order, NaN above Inf); each CTA issues one atomicMax
// per copy into the two output floats, which the host wrapper zeroes first.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tile_pipeline.cuh"

namespace nvfp4 {
namespace {

using tile::kTM;
using tile::kTN;
constexpr int kBlockThreads = 256;

__device__ __forceinline__ uint32_t absmax_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// packed bf16 |max| -> float bits of the larger half (sign dropped)
__device__ __forceinline__ uint32_t packed_to_bits(uint32_t m) {
  m &= 0x7FFF7FFFu;
  return max(m << 16, m & 0xFFFF0000u);
}

// NaN-propagating maximum of m and |v| (for non-negative m, the same order as
// the bit patterns of the magnitudes: NaN above Inf above every finite value)
__device__ __forceinline__ float max_abs_nan(float m, float v) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(v)));
  return r;
}

// CTA-wide max of two values, then one atomicMax each.
__device__ __forceinline__ void cta_reduce_and_publish(uint32_t vr, uint32_t vc, float* amax) {
  __shared__ uint32_t red[2][kBlockThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  vr = __reduce_max_sync(0xFFFFFFFFu, vr);
  vc = __reduce_max_sync(0xFFFFFFFFu, vc);
  if (lane == 0) {
    red[0][warp] = vr;
    red[1][warp] = vc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t br = 0u, bc = 0u;
#pragma unroll
    for (int w = 0; w < kBlockThreads / 32; ++w) {
      br = max(br, red[0][w]);
      bc = max(bc, red[1][w]);
    }
    atomicMax(reinterpret_cast<unsigned int*>(amax), br);
    atomicMax(reinterpret_cast<unsigned int*>(amax) + 1, bc);
  }
}

__global__ void __launch_bounds__(kBlockThreads) amax_flat_kernel(const uint4* x, int64_t nchunks, float* amax) {
  constexpr int U = 4;
  uint32_t m = 0u;
  const int64_t stride = (int64_t)gridDim.x * kBlockThreads * U;
  for (int64_t base = (int64_t)blockIdx.x * kBlockThreads * U + threadIdx.x; base < nchunks; base += stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + (int64_t)u * kBlockThreads;
      v[u] = (i < nchunks) ? ld_stream(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      m = absmax_nan_bf16x2(m, absmax_nan_bf16x2(absmax_nan_bf16x2(v[u].x, v[u].y),
                                                 absmax_nan_bf16x2(v[u].z, v[u].w)));
  }
  const uint32_t bits = packed_to_bits(m);
  cta_reduce_and_publish(bits, bits, amax);
}

template <bool RHT_ROW, bool RHT_COL>
__global__ void __launch_bounds__(kBlockThreads) amax_tile_kernel(const AmaxArgs a) {
  extern __shared__ __align__(16) uint8_t bufs[];  // 2 x 32 KB tiles
  const int64_t M = a.M, N = a.N;
  const int tid = threadIdx.x;
  const uint32_t signs = (RHT_ROW || RHT_COL) ? rht_sign_bits(a.rht_k0, a.rht_k1) : 0u;
  const int rb_b = tid & 15, rb_r0 = tid >> 4;    // rowwise tasks
  const int cp_p = tid & 127, cp_rb0 = tid >> 7;  // columnwise tasks
  uint32_t m_plain = 0u;
  float m_row = 0.0f, m_col = 0.0f;

  tile::Walker w;
  w.init(M, N);
  if (w.valid()) tile::load_async<kBlockThreads>(bufs, a.x, M, N, a.ld, w.coord(), tid);
  tile::commit();
  for (int it = 0; w.valid(); w = w.next(), ++it) {
    const uint8_t* buf = bufs + (it & 1) * tile::kTileBytes;
    const tile::Walker wn = w.next();
    if (wn.valid())
      tile::load_async<kBlockThreads>(bufs + ((it + 1) & 1) * tile::kTileBytes, a.x, M, N, a.ld, wn.coord(), tid);
    tile::commit();
    tile::wait_all_but_one();
    __syncthreads();
    const tile::Coord tc = w.coord();
    const int rows = (int)((M - tc.R0) < kTM ? (M - tc.R0) : kTM);
    const int cols = (int)((N - tc.C0) < kTN ? (N - tc.C0) : kTN);
    if (RHT_COL || !RHT_ROW) {
      // columnwise tasks: plain max of every element, and the transformed
      // column vectors' max when the columnwise copy has the RHT
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int rb = cp_rb0 + 2 * k;
        if (2 * cp_p >= cols || 16 * rb >= rows) continue;
        uint32_t wd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) wd[i] = tile::read_pair_word(buf, 16 * rb + i, cp_p);
#pragma unroll
        for (int i = 0; i < 16; i += 2) m_plain = absmax_nan_bf16x2(m_plain, absmax_nan_bf16x2(wd[i], wd[i + 1]));
        if (RHT_COL) {  // both columns at once; the 1/4 is applied to the maximum
          float2 zp[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) zp[i] = bf16x2_to_f32x2(wd[i] ^ rht_mask_col(signs, i));
          wht16_x2(zp);
#pragma unroll
          for (int i = 0; i < 16; ++i) m_col = max_abs_nan(max_abs_nan(m_col, zp[i].x), zp[i].y);
        }
      }
    }
    if (RHT_ROW) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int r = rb_r0 + 16 * k;
        if (16 * rb_b >= cols || r >= rows) continue;
        uint32_t wd[8];
        tile::read_row_block(buf, r, rb_b, wd);
        if (!RHT_COL) {
#pragma unroll
          for (int i = 0; i < 8; i += 2) m_plain = absmax_nan_bf16x2(m_plain, absmax_nan_bf16x2(wd[i], wd[i + 1]));
        }
        float z[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = bf16x2_to_f32x2(wd[j] ^ rht_mask_row(signs, j));
          z[2 * j] = f.x;
          z[2 * j + 1] = f.y;
        }
        wht16(z);
#pragma unroll
        for (int j = 0; j < 16; ++j) m_row = max_abs_nan(m_row, z[j]);
      }
    }
    __syncthreads();  // the buffer is refilled by the next iteration's prefetch
  }
  const uint32_t plain = packed_to_bits(m_plain);
  // max |y| = max |t| / 4 for the unnormalised butterfly output t: the scaling
  // is exact and rounding is monotonic, so it commutes with the maximum
  const uint32_t quarter_row = __float_as_uint(__fmul_rn(m_row, 0.25f));
  const uint32_t quarter_col = __float_as_uint(__fmul_rn(m_col, 0.25f));
  cta_reduce_and_publish(RHT_ROW ? quarter_row : plain, RHT_COL ? quarter_col : plain, a.amax);
}

template <bool RHT_ROW, bool RHT_COL>
cudaError_t launch_tile(const AmaxArgs& a, cudaStream_t s) {
  constexpr int kSmem = 2 * tile::kTileBytes;
  auto kern = amax_tile_kernel<RHT_ROW, RHT_COL>;
  static std::atomic<int> grid_cap[64] = {};
  int cap = 0;
  const cudaError_t ge = resident_grid(kern, kBlockThreads, kSmem, grid_cap, cap);
  if (ge != cudaSuccess) return ge;
  const int64_t ntiles = ((a.M + kTM - 1) / kTM) * ((a.N + kTN - 1) / kTN);
  int64_t g = ntiles < cap ? ntiles : cap;
  if (g < 1) g = 1;
  kern<<<(unsigned)g, kBlockThreads, kSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_amax(const AmaxArgs& a, bool rht_row, bool rht_col, cudaStream_t s) {
  if (!rht_row && !rht_col && a.ld == a.N) {
    const int64_t nchunks = a.M * a.N / 8;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t grid = (nchunks + kBlockThreads * 4 - 1) / (kBlockThreads * 4);
    if (grid > (int64_t)sms * 8) grid = (int64_t)sms * 8;
    if (grid < 1) grid = 1;
    amax_flat_kernel<<<(unsigned)grid, kBlockThreads, 0, s>>>(reinterpret_cast<const uint4*>(a.x), nchunks,
                                                              a.amax);
    return cudaGetLastError();
  }
  if (rht_row && rht_col) return launch_tile<true, true>(a, s);
  if (rht_row) return launch_tile<true, false>(a, s);
  if (rht_col) return launch_tile<false, true>(a, s);
  return launch_tile<false, false>(a, s);
}

}  // namespace nvfp4
