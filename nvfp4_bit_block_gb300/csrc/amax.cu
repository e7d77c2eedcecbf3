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
//     quantize kernel's 64 x 256 shared-memory tile and its two passes.
// Maxima are combined as the bit patterns of non-negative floats (unsigned
// order equals float order, NaN above Inf); each CTA issues one atomicMax
// per copy into the two output floats, which the host wrapper zeroes first.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kTM = 64, kTN = 256, kRowBytes = kTN * 2, kBlockThreads = 256;

__device__ __forceinline__ int swz_tile(int c) { return c ^ ((c >> 3) & 1); }

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

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

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
  __shared__ __align__(16) uint8_t tile[kTM * kRowBytes];
  const int64_t M = a.M, N = a.N;
  const int64_t R0 = (int64_t)blockIdx.y * kTM, C0 = (int64_t)blockIdx.x * kTN;
  const int tid = threadIdx.x;
  uint32_t m = 0u;
  {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int id = tid + k * kBlockThreads;
      const int r = id >> 5, c = id & 31;
      const int64_t grow = R0 + r, gcol = C0 + 8 * c;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (grow < M && gcol < N) v[k] = ld_stream(a.x + grow * a.ld + gcol);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      m = absmax_nan_bf16x2(m, absmax_nan_bf16x2(absmax_nan_bf16x2(v[k].x, v[k].y),
                                                 absmax_nan_bf16x2(v[k].z, v[k].w)));
      if (RHT_ROW || RHT_COL) {
        const int id = tid + k * kBlockThreads;
        const int r = id >> 5, c = id & 31;
        *reinterpret_cast<uint4*>(tile + r * kRowBytes + swz_tile(c) * 16) = v[k];
      }
    }
  }
  const uint32_t plain = packed_to_bits(m);
  uint32_t m_row = 0u, m_col = 0u;
  if (RHT_ROW || RHT_COL) {
    __syncthreads();
    const uint32_t signs = rht_sign_bits(a.rht_k0, a.rht_k1);
    if (RHT_ROW) {
#pragma unroll 1
      for (int k = 0; k < kTM * 16 / kBlockThreads; ++k) {
        const int task = tid + k * kBlockThreads;
        const int r = task >> 4, b = task & 15;
        if (R0 + r >= M || C0 + 16 * b >= N) continue;
        const uint4 lo = *reinterpret_cast<const uint4*>(tile + r * kRowBytes + swz_tile(2 * b) * 16);
        const uint4 hi = *reinterpret_cast<const uint4*>(tile + r * kRowBytes + swz_tile(2 * b + 1) * 16);
        const uint32_t wd[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        float z[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          z[2 * j] = bf16_lo(wd[j]);
          z[2 * j + 1] = bf16_hi(wd[j]);
        }
        rht16(z, signs);
#pragma unroll
        for (int j = 0; j < 16; ++j) m_row = max(m_row, abs_bits(z[j]));
      }
    }
    if (RHT_COL) {
#pragma unroll 1
      for (int k = 0; k < (kTN / 2) * (kTM / 16) / kBlockThreads; ++k) {
        const int task = tid + k * kBlockThreads;
        const int p = task & 127, rb = task >> 7;
        if (C0 + 2 * p >= N || R0 + 16 * rb >= M) continue;
        uint32_t wd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wd[i] = *reinterpret_cast<const uint32_t*>(tile + (16 * rb + i) * kRowBytes + swz_tile(p >> 2) * 16 +
                                                     (p & 3) * 4);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          float z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = h ? bf16_hi(wd[i]) : bf16_lo(wd[i]);
          rht16(z, signs);
#pragma unroll
          for (int i = 0; i < 16; ++i) m_col = max(m_col, abs_bits(z[i]));
        }
      }
    }
  }
  cta_reduce_and_publish(RHT_ROW ? m_row : plain, RHT_COL ? m_col : plain, a.amax);
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
  const int64_t gx = (a.N + kTN - 1) / kTN, gy = (a.M + kTM - 1) / kTM;
  const dim3 grid((unsigned)gx, (unsigned)gy, 1);
  if (rht_row && rht_col)
    amax_tile_kernel<true, true><<<grid, kBlockThreads, 0, s>>>(a);
  else if (rht_row)
    amax_tile_kernel<true, false><<<grid, kBlockThreads, 0, s>>>(a);
  else if (rht_col)
    amax_tile_kernel<false, true><<<grid, kBlockThreads, 0, s>>>(a);
  else
    amax_tile_kernel<false, false><<<grid, kBlockThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
