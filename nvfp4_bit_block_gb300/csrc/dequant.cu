// dequant.cu -- x^ = val(code) * (float(e) * alpha), fp32 or bf16 output.
//
// The reconstruction the 4/6 error of the "Four Over Six (4/6)" technical
// summary (Methodology, step 2) is measured against.  One thread decodes one
// 16-element block: an 8-byte code load, one scale byte, 64 bytes (fp32) or
// 32 bytes (bf16) of vector stores.
#include <cuda_bf16.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

__global__ void __launch_bounds__(256) dequant_kernel(const DequantArgs a) {
  const int64_t blocks_per_row = a.cols / 16;
  const int64_t nblocks = a.rows * blocks_per_row;
  const float alpha = *a.alpha;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblocks;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = blk / blocks_per_row;
    const int64_t kb = blk - r * blocks_per_row;
    const uint2 codes = *reinterpret_cast<const uint2*>(a.q + r * (a.cols / 2) + kb * 8);
    const float d = __fmul_rn(e4m3_value(a.s[r * blocks_per_row + kb]), alpha);
    float out[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t word = (j < 4) ? codes.x : codes.y;
      const float2 v = e2m1x2_values((word >> (8 * (j & 3))) & 0xFFu);
      out[2 * j] = __fmul_rn(v.x, d);
      out[2 * j + 1] = __fmul_rn(v.y, d);
    }
    if (a.out_bf16) {
      uint32_t p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(out[2 * j], out[2 * j + 1]);
        p[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + r * a.cols + kb * 16);
      dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
      dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + r * a.cols + kb * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s) {
  const int64_t nblocks = a.rows * (a.cols / 16);
  int64_t grid = (nblocks + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;  // grid-stride beyond 32 CTAs per SM
  if (grid < 1) grid = 1;
  dequant_kernel<<<(unsigned)grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
