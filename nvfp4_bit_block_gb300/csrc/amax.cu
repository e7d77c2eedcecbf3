// amax.cu -- tensor amax for the rowwise and the columnwise copy.
//
// "Four Over Six (4/6)" technical summary, Implementation details: the global
// tensor scale comes from the tensor's largest magnitude.  A copy that is
// Hadamard-transformed ("Pretraining Large Language Models with NVFP4"
// section 2b) takes the largest magnitude of its transformed 16-vectors,
// computed with exactly the butterfly the quantize kernel uses, so the scale
// always covers the values that are quantized.
//
// Maxima are taken on the bit patterns of non-negative floats (which order
// like unsigned integers, with NaN above Inf), so a NaN input propagates to
// the result.  Each CTA reduces in shared memory and issues one atomicMax per
// copy; the two output floats are zeroed by the host wrapper beforehand.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

template <bool RHT_ROW, bool RHT_COL>
__global__ void __launch_bounds__(kThreads) amax_kernel(const AmaxArgs a) {
  __shared__ uint32_t red[2][kWarps];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool odd = (lane & 1) != 0;
  const int64_t r0 = ((int64_t)blockIdx.y * kWarps + warp) * 16;
  const int64_t c0 = (int64_t)blockIdx.x * kTileCols + lane * 8;
  const bool col_ok = c0 < a.N;
  const bool warp_ok = r0 < a.M;

  uint32_t m_plain = 0u, m_row = 0u, m_col = 0u;
  if (warp_ok) {  // warp-uniform
    uint32_t xr[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok && r0 + i < a.M) v = ld_stream(a.x + (r0 + i) * a.ld + c0);
      xr[i][0] = v.x;
      xr[i][1] = v.y;
      xr[i][2] = v.z;
      xr[i][3] = v.w;
    }
    // plain max over |bf16| bit patterns (15 bits, unsigned order = float order)
    uint32_t mlo = 0u, mhi = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mlo = max(mlo, xr[i][k] & 0x7FFFu);
        mhi = max(mhi, (xr[i][k] >> 16) & 0x7FFFu);
      }
    m_plain = max(mlo, mhi) << 16;
    if (RHT_ROW || RHT_COL) {
      const uint32_t signs = rht_sign_bits(a.rht_k0, a.rht_k1);
      if (RHT_ROW) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float z[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            z[2 * k] = bf16_lo(xr[i][k]);
            z[2 * k + 1] = bf16_hi(xr[i][k]);
          }
          rht16_pair(z, signs, odd);
#pragma unroll
          for (int j = 0; j < 8; ++j) m_row = max(m_row, abs_bits(z[j]));
        }
      }
      if (RHT_COL) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = (cc & 1) ? bf16_hi(xr[i][cc >> 1]) : bf16_lo(xr[i][cc >> 1]);
          rht16(z, signs);
#pragma unroll
          for (int i = 0; i < 16; ++i) m_col = max(m_col, abs_bits(z[i]));
        }
      }
    }
  }
  const uint32_t out_r = RHT_ROW ? m_row : m_plain;
  const uint32_t out_c = RHT_COL ? m_col : m_plain;
  const uint32_t wr = __reduce_max_sync(0xFFFFFFFFu, out_r);
  const uint32_t wc = __reduce_max_sync(0xFFFFFFFFu, out_c);
  if (lane == 0) {
    red[0][warp] = wr;
    red[1][warp] = wc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t br = 0u, bc = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      br = max(br, red[0][w]);
      bc = max(bc, red[1][w]);
    }
    atomicMax(reinterpret_cast<unsigned int*>(a.amax), br);
    atomicMax(reinterpret_cast<unsigned int*>(a.amax) + 1, bc);
  }
}

}  // namespace

cudaError_t launch_amax(const AmaxArgs& a, bool rht_row, bool rht_col, cudaStream_t s) {
  const dim3 grid = tile_grid(a.M, a.N);
  if (rht_row && rht_col)
    amax_kernel<true, true><<<grid, kThreads, 0, s>>>(a);
  else if (rht_row)
    amax_kernel<true, false><<<grid, kThreads, 0, s>>>(a);
  else if (rht_col)
    amax_kernel<false, true><<<grid, kThreads, 0, s>>>(a);
  else
    amax_kernel<false, false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
