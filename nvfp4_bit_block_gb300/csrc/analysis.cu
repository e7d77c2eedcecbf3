// analysis.cu -- quantization-error histogram of a rowwise copy over the
// scaled value.
//
// "Four Over Six (4/6)" technical summary, Problem statement: with the block
// maximum scaled to 6, values between 4 and 6 (66.6-100 % of the block max)
// fall in the grid's widest gap, and the rounding error around scaled value 5
// -- rather than the error of the scale factors -- is what degrades quantized
// models.  This tool measures that on a tensor and one of its quantizations.
// Each element's position in its block, v = 6|x| / b (b = the block's largest
// magnitude, so v is in [0, 6]), selects one of nbins equal bins over [0, 6]
// (bin = min(floor(v * nbins / 6), nbins - 1)); the bin accumulates the
// element count, the sum of e = 6|x - x^| / b (x^ = the dequantized value,
// computed as nvfp4_dequantize does) and the sum of e * e.  Sums are fixed
// point (e in units of 2^-24, e * e in units of 2^-32, each term truncated),
// so the totals are exact integers whatever the order of accumulation.
// Blocks whose maximum is 0 are skipped.  All steps are single IEEE
// round-to-nearest operations in the order written.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) error_hist_kernel(const HistArgs a) {
  extern __shared__ unsigned long long hist[];  // [3][nbins]
  const int nb = a.nbins;
  for (int i = threadIdx.x; i < 3 * nb; i += kThreads) hist[i] = 0ull;
  __syncthreads();
  const int64_t bpr = a.N / 16;
  const int64_t nblocks = a.M * bpr;
  const float alpha = *a.alpha;
  const float fnb = (float)nb;
  for (int64_t blk = (int64_t)blockIdx.x * kThreads + threadIdx.x; blk < nblocks;
       blk += (int64_t)gridDim.x * kThreads) {
    const int64_t r = blk / bpr, kb = blk - r * bpr;
    const uint4* xp = reinterpret_cast<const uint4*>(a.x + r * a.ld + kb * 16);
    const uint4 lo = xp[0], hi = xp[1];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const float b = block_absmax16(w);
    if (!(b > 0.0f)) continue;
    const uint2 codes = *reinterpret_cast<const uint2*>(a.q + r * (a.N / 2) + kb * 8);
    const float d = __fmul_rn(e4m3_value(a.s[r * bpr + kb]), alpha);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float x = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
      const uint32_t word = (j < 8) ? codes.x : codes.y;
      const float2 vals = e2m1x2_values((word >> (8 * ((j >> 1) & 3))) & 0xFFu);
      const float xh = __fmul_rn((j & 1) ? vals.y : vals.x, d);
      const float v = __fdiv_rn(__fmul_rn(6.0f, fabsf(x)), b);
      int bin = (int)floorf(__fdiv_rn(__fmul_rn(v, fnb), 6.0f));
      bin = bin < nb - 1 ? bin : nb - 1;
      const float e = __fdiv_rn(__fmul_rn(6.0f, fabsf(__fsub_rn(x, xh))), b);
      atomicAdd(&hist[bin], 1ull);
      atomicAdd(&hist[nb + bin], __float2ull_rz(__fmul_rn(e, 0x1p24f)));
      atomicAdd(&hist[2 * nb + bin], __float2ull_rz(__fmul_rn(__fmul_rn(e, e), 0x1p32f)));
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 3 * nb; i += kThreads)
    if (hist[i]) atomicAdd(a.hist + i, hist[i]);
}

}  // namespace

cudaError_t launch_error_hist(const HistArgs& a, cudaStream_t s) {
  const int64_t nblocks = a.M * (a.N / 16);
  int64_t grid = (nblocks + kThreads - 1) / kThreads;
  if (grid > 152 * 8) grid = 152 * 8;
  if (grid < 1) grid = 1;
  error_hist_kernel<<<(unsigned)grid, kThreads, 3 * a.nbins * sizeof(unsigned long long), s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
