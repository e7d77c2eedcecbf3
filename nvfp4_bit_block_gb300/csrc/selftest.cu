// selftest.cu -- exhaustive device check of the scale-byte quotient.
//
// The quantize kernels take E4M3(fl(b / den)) from scale_byte (quotient_rn:
// a product and one residual correction, capped at 1e6) instead of an IEEE
// division.  This kernel compares the two bytes for every pair of a bf16
// block maximum b (any finite value: an amax supplied by the caller may be
// smaller than the block) and a bf16 tensor amax A that the library accepts
// (2^-100 <= A finite), with den = Q * (A / 2688) for Q = 6 and
// den = Q * (A / 1536) for Q = 6 and 4, exactly as the kernels form them; the
// same again with A replaced by a pseudo-random fp32 value just above it (an
// amax that is not a bf16 value, e.g. of a transformed copy); and 256
// pseudo-random fp32 maxima in [0, 4A) per (A, den), as a transformed
// (Hadamard) block has.  It reports how many scale bytes differ, how many
// quotients differ where the IEEE quotient is a normal fp32 number below the
// cap, how many differ at all, and the first differing byte case.
#include <cstdint>

#include "nvfp4.h"
#include "nvfp4_device.cuh"

namespace nvfp4 {
namespace {

constexpr uint32_t kFirstA = 0x0D80u;  // bf16 bits of 2^-100
constexpr uint32_t kLastA = 0x7F7Fu;   // largest finite bf16

__device__ __forceinline__ uint32_t mix32(uint32_t x) {  // a 32-bit integer hash (xorshift-multiply)
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return x;
}

// out[0] = differing bytes, out[1] = differing normal quotients,
// out[2] = first differing byte case: (grid y << 32) | (A bits << 16) | b bits,
// out[3] = differing quotients of any size, out[4] / out[5] = differing bytes
// with a second correction / with the bare product b * rden
__global__ void quotient_check_kernel(unsigned long long* out) {
  const uint32_t abits = kFirstA + blockIdx.x;
  const int combo = blockIdx.y % 3;  // 0: Q=6 over 2688; 1: Q=6 over 1536; 2: Q=4 over 1536
  float A = __uint_as_float(abits << 16);
  if (blockIdx.y >= 3) {  // an fp32 amax between this bf16 value and the next
    const uint32_t h = mix32(abits * 0x2545F491u + blockIdx.y);
    A = __uint_as_float((abits << 16) | (h & 0xFFFFu));
  }
  const float alpha = __fdiv_rn(A, combo == 0 ? kAlphaDen : kAlphaDen46);
  const float den = __fmul_rn(combo == 2 ? 4.0f : 6.0f, alpha);
  const float rden = (den != 0.0f) ? __frcp_rn(den) : 0.0f;
  unsigned long long bytes = 0, quots = 0, quots_all = 0, bytes1 = 0, bytes0 = 0;
  for (uint32_t bb = threadIdx.x; bb <= kLastA + 256u; bb += blockDim.x) {
    float b;
    if (bb <= kLastA) {
      b = __uint_as_float(bb << 16);
    } else {  // random fp32 in [0, 4A)
      const uint32_t h = mix32(abits * 0x9E3779B9u + blockIdx.y * 0x85EBCA6Bu + bb);
      b = __fmul_rn(A, __fmul_rn((float)(h >> 8), 0x1p-22f));
    }
    const float q = quotient_rn(b, den, rden);
    const float ref = __fdiv_rn(b, den);
    const uint32_t eref = e4m3_encode(ref);
    if (__float_as_uint(q) != __float_as_uint(ref) && ref < 1.0e6f) {
      ++quots_all;
      if (ref >= 0x1p-126f) ++quots;
    }
    {  // a second correction, and the bare product, for comparison
      const float r2 = __fmaf_rn(-q, den, b);
      const float q2 = __fmaf_rn(r2, rden, q);
      if (e4m3_encode(fminf(q2, 1.0e6f)) != eref) ++bytes1;
      if (e4m3_encode(__fmul_rn(b, rden)) != eref) ++bytes0;
    }
    if (scale_byte(b, den, rden) != eref) {
      ++bytes;
      atomicCAS(out + 2, 0ull,
                ((unsigned long long)blockIdx.y << 32) | ((unsigned long long)abits << 16) | (bb & 0xFFFFu));
    }
  }
  if (bytes) atomicAdd(out + 0, bytes);
  if (quots) atomicAdd(out + 1, quots);
  if (quots_all) atomicAdd(out + 3, quots_all);
  if (bytes1) atomicAdd(out + 4, bytes1);
  if (bytes0) atomicAdd(out + 5, bytes0);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

// Test hook (not declared in nvfp4.h): run the exhaustive quotient check.
// out_dev: six zeroed unsigned 64-bit counters on the device (see above).
NVFP4_API int nvfp4_test_quotient_check(unsigned long long* out_dev, void* stream) {
  if (!out_dev) return NVFP4_ERR_NULL;
  const dim3 grid(nvfp4::kLastA - nvfp4::kFirstA + 1, 6);
  nvfp4::quotient_check_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(out_dev);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"
