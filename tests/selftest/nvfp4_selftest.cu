// nvfp4_selftest.cu -- device self-checks of the quantizer's building blocks,
// built into a test-only library (libnvfp4_selftest.so) that the tests load;
// the product library holds none of this code.
//
// Exhaustive device check of the scale-byte quotient.
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
//
// A second hook runs the kernels' Hadamard transform alone, so that the
// transformed values themselves can be compared with a reference.  A third
// compares the kernels' Philox4x32-10 (the stochastic-rounding words and the
// RHT sign word) with cuRAND's device implementation of the same generator,
// an independent one, over pseudo-random and extreme counters and keys.  A
// fourth launches a 1D quantize kernel (round-to-nearest, or stochastic
// rounding on both copies) in a variant that arms its tile barriers but
// issues no copy, so that the bounded wait runs out.  A fifth
// runs the kernels' stochastic rounding alone on given values and words, and
// a sixth launches the GEMM in a variant whose copies are never issued.
#include <cstdint>

#include <curand_philox4x32_x.h>

#include "nvfp4.h"
#include "nvfp4_device.cuh"
#include "gemm_kernel.cuh"
#include "quant1d_kernel.cuh"
#include "quant1d_sr_kernel.cuh"

namespace {
bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
}  // namespace

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
  if (!aligned(out_dev, 8)) return NVFP4_ERR_ALIGN;
  const dim3 grid(nvfp4::kLastA - nvfp4::kFirstA + 1, 6);
  nvfp4::quotient_check_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(out_dev);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The kernels' 16-point random Hadamard transform, alone: out (fp32, M x N)
// holds y = (1/4) H16 (s . x) of every 16-vector along rows (along_cols = 0)
// or along columns (along_cols = 1), formed with the same masks and packed
// butterflies as the quantize kernels (one thread per vector pair).
__global__ void rht_check_kernel(const uint16_t* x, int64_t M, int64_t N, int64_t ld, int along_cols,
                                 uint32_t k0, uint32_t k1, float* out) {
  const uint32_t signs = rht_sign_bits(k0, k1);
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (!along_cols) {  // one rowwise vector per thread
    const int64_t nv = M * (N / 16);
    if (t >= nv) return;
    const int64_t r = t / (N / 16), c0 = (t - r * (N / 16)) * 16;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(x + r * ld + c0);
    float z[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = bf16x2_to_f32x2(w[j] ^ rht_mask_row(signs, j));
      z[2 * j] = f.x;
      z[2 * j + 1] = f.y;
    }
    wht16(z);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[r * N + c0 + j] = __fmul_rn(z[j], 0.25f);
  } else {  // two columnwise vectors (columns 2p, 2p+1, rows 16b..16b+15) per thread
    const int64_t nv = (M / 16) * (N / 2);
    if (t >= nv) return;
    const int64_t b = t / (N / 2), p = t - b * (N / 2);
    float2 zp[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(x + (16 * b + i) * ld + 2 * p);
      zp[i] = bf16x2_to_f32x2(w ^ rht_mask_col(signs, i));
    }
    wht16_x2(zp);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 y = mul2(zp[i], make_float2(0.25f, 0.25f));
      out[(16 * b + i) * N + 2 * p] = y.x;
      out[(16 * b + i) * N + 2 * p + 1] = y.y;
    }
  }
}

}  // namespace
}  // namespace nvfp4

extern "C" {

// Test hook (not declared in nvfp4.h): the kernels' Hadamard transform of a
// bf16 M x N tensor (row stride ld, 4-byte aligned rows), 16-vectors along
// rows or columns, into a dense fp32 M x N buffer (4-byte aligned).
NVFP4_API int nvfp4_test_rht(const void* x_dev, int64_t M, int64_t N, int64_t ld, int along_cols, uint64_t rht_seed,
                             float* out_dev, void* stream) {
  if (!x_dev || !out_dev) return NVFP4_ERR_NULL;
  if (M <= 0 || N <= 0 || N % 16 || ld < N || (along_cols && M % 16)) return NVFP4_ERR_SHAPE;
  if (ld % 2 || !aligned(x_dev, 4) || !aligned(out_dev, 4)) return NVFP4_ERR_ALIGN;
  const int64_t nv = along_cols ? (M / 16) * (N / 2) : M * (N / 16);
  const int64_t grid = (nv + 255) / 256;
  nvfp4::rht_check_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x_dev), M, N, ld, along_cols, (uint32_t)rht_seed, (uint32_t)(rht_seed >> 32),
      out_dev);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"

namespace nvfp4 {
namespace {

// out[0] = counters whose words 0/1 differ from cuRAND's, out[1] = keys whose
// 16 RHT sign bits (low half of word 0) differ, out[2] = cases checked,
// out[3] = counters where the form with the second-round product given
// differs, out[4] = words of 16-counter blocks that differ, out[5] = blocks
// checked that cross a multiple of 2^32.  Thread t of the grid takes
// counter (c0, c1) and key (k0, k1) from a hash of t; the first 4096 threads
// take counter and key words from {0, 1, 2^31, 2^32 - 1} instead, so that
// carries and all-ones words are covered.
__global__ void philox_check_kernel(unsigned long long* out) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t c0, c1, k0, k1;
  if (t < 4096u) {
    const uint32_t ext[4] = {0u, 1u, 0x80000000u, 0xFFFFFFFFu};
    c0 = ext[t & 3u];
    c1 = ext[(t >> 2) & 3u];
    k0 = ext[(t >> 4) & 3u];
    k1 = ext[(t >> 6) & 3u];
    if (t >= 256u) {  // the rest: one extreme word, the others hashed
      c0 ^= mix32(t * 0x9E3779B9u) & ((t >> 8) & 1u ? 0xFFFFFFFFu : 0u);
      c1 ^= mix32(t * 0x85EBCA6Bu) & ((t >> 9) & 1u ? 0xFFFFFFFFu : 0u);
      k0 ^= mix32(t * 0xC2B2AE35u) & ((t >> 10) & 1u ? 0xFFFFFFFFu : 0u);
      k1 ^= mix32(t * 0x27D4EB2Fu) & ((t >> 11) & 1u ? 0xFFFFFFFFu : 0u);
    }
  } else {
    c0 = mix32(t * 0x9E3779B9u + 1u);
    c1 = mix32(t * 0x85EBCA6Bu + 2u);
    k0 = mix32(t * 0xC2B2AE35u + 3u);
    k1 = mix32(t * 0x27D4EB2Fu + 4u);
  }
  const uint2 ours = philox_w01(c0, c1, k0, k1);
  const uint4 ref = curand_Philox4x32_10(make_uint4(c0, c1, 0u, 0u), make_uint2(k0, k1));
  if (ours.x != ref.x || ours.y != ref.y) atomicAdd(out + 0, 1ull);
  // the form with the second-round product given, and the 16-counter form
  // (stride 1 or a hashed stride; the extreme words make blocks that cross a
  // multiple of 2^32)
  const uint2 sh = philox_w01_shared_hi(c0, (uint64_t)0xD2511F53u * (c1 ^ k0), k0, k1);
  if (sh.x != ref.x || sh.y != ref.y) atomicAdd(out + 3, 1ull);
  const uint32_t stride = (t & 1u) ? 1u : (mix32(t * 0x165667B1u) >> 12);
  const uint64_t base = (((uint64_t)c1 << 32) | c0) - ((t & 2u) ? 7ull * stride : 0ull);
  uint32_t w0[16], w1[16];
  philox_group_w01<16, true>(base, stride, k0, k1, w0, w1);
  unsigned long long bad16 = 0;
#pragma unroll 1
  for (int j = 0; j < 16; ++j) {
    const uint64_t i = base + (uint64_t)j * stride;
    const uint4 r = curand_Philox4x32_10(make_uint4((uint32_t)i, (uint32_t)(i >> 32), 0u, 0u), make_uint2(k0, k1));
    if (w0[j] != r.x || w1[j] != r.y) ++bad16;
  }
  if (bad16) atomicAdd(out + 4, bad16);
  if ((base >> 32) != ((base + 15ull * stride) >> 32)) atomicAdd(out + 5, 1ull);
  const uint4 ref_sign = curand_Philox4x32_10(make_uint4(0u, 0u, 0u, 1u), make_uint2(k0, k1));
  if (rht_sign_bits(k0, k1) != (ref_sign.x & 0xFFFFu)) atomicAdd(out + 1, 1ull);  // 16 signs: low half of word 0
  atomicAdd(out + 2, 1ull);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

// Test hook (not declared in nvfp4.h): compare the kernels' Philox4x32-10 with
// cuRAND's over `blocks` x 256 counter/key cases (blocks >= 16 covers the
// extreme words).  out_dev: six zeroed unsigned 64-bit counters (see above).
NVFP4_API int nvfp4_test_philox_check(unsigned long long* out_dev, int blocks, void* stream) {
  if (!out_dev) return NVFP4_ERR_NULL;
  if (!aligned(out_dev, 8)) return NVFP4_ERR_ALIGN;
  if (blocks <= 0) return NVFP4_ERR_SHAPE;
  nvfp4::philox_check_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(out_dev);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"

extern "C" {

// Test hook: a rowwise + columnwise 1D quantize kernel in a variant whose
// tile barriers are armed but whose copies are never issued, so every wait
// runs out: the kernel writes NVFP4_ERR_PIPELINE to status_dev after about a
// second and returns.  sr = 0: the round-to-nearest kernel (flags ROWWISE |
// COLWISE); sr = 1: the stochastic-rounding kernel (ROWWISE | COLWISE | SR).
// Other arguments as nvfp4_quantize; all pointers are required.
NVFP4_API int nvfp4_test_quantize_no_copy(const void* x_dev, int64_t M, int64_t N, int64_t ld, const float* amax_dev,
                                          uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                          float* alpha_dev, int* status_dev, int sr, void* stream) {
  if (!x_dev || !amax_dev || !q_row || !s_row || !q_col || !s_col || !alpha_dev || !status_dev) return NVFP4_ERR_NULL;
  if (M <= 0 || N <= 0 || M % 16 || N % 16 || ld < N || M > INT32_MAX || N > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (ld % 8 || !aligned(x_dev, 16) || !aligned(q_row, 16) || !aligned(q_col, 16) || !aligned(s_row, 4) ||
      !aligned(s_col, 4) || !aligned(amax_dev, 4) || !aligned(alpha_dev, 4) || !aligned(status_dev, 4))
    return NVFP4_ERR_ALIGN;
  nvfp4::QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x_dev);
  a.M = M;
  a.N = N;
  a.ld = ld;
  a.amax = amax_dev;
  a.alpha = alpha_dev;
  a.status = status_dev;
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.sel = nvfp4::kSelMAE;
  if (sr != 0 && sr != 1) return NVFP4_ERR_FLAGS;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = sr ? nvfp4::q1d::launch_sr_rc<false, true>(a, s)
                           : nvfp4::q1d::launch<true, true, false, false, nvfp4::kSelMAE, 0, true>(a, s);
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The kernels' stochastic rounding alone: out[i] = sr_round(v[i], Q, w[i]).
__global__ void sr_round_kernel(const float* v, const uint32_t* w, int64_t n, float Q, float* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = sr_round(v[i], Q, w[i]);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

// Test hook: run the kernels' stochastic rounding onto the E2M1 grid (block
// maximum Q = 6 or 4) on n values v with random words w; out receives the
// signed grid values.  All arrays are fp32 / uint32 on the device.
NVFP4_API int nvfp4_test_sr_round(const float* v_dev, const uint32_t* w_dev, int64_t n, float Q, float* out_dev,
                                  void* stream) {
  if (!v_dev || !w_dev || !out_dev) return NVFP4_ERR_NULL;
  if (n < 0 || (Q != 6.0f && Q != 4.0f)) return NVFP4_ERR_SHAPE;
  if (!aligned(v_dev, 4) || !aligned(w_dev, 4) || !aligned(out_dev, 4)) return NVFP4_ERR_ALIGN;
  if (n == 0) return NVFP4_OK;
  const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  nvfp4::sr_round_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(v_dev, w_dev, n, Q,
                                                                                          out_dev);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"

extern "C" {

// Test hook: the NVFP4 GEMM in a variant whose producer arms the stage
// barriers but issues no copy, so every wait runs out: the kernel writes
// NVFP4_ERR_PIPELINE to status_dev after about a second, drains and frees its
// tensor memory, and returns.  Arguments as nvfp4_gemm; all pointers are
// required.
NVFP4_API int nvfp4_test_gemm_no_copy(const uint8_t* qa, const uint8_t* sfa, const float* alpha_a, const uint8_t* qb,
                                      const uint8_t* sfb, const float* alpha_b, void* d, int64_t M, int64_t N,
                                      int64_t K, int64_t ldd, int out_bf16, int* status_dev, void* stream) {
  if (!qa || !sfa || !alpha_a || !qb || !sfb || !alpha_b || !d || !status_dev) return NVFP4_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 256 || ldd < N) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sfa, 16) || !aligned(sfb, 16) || !aligned(d, 16) ||
      !aligned(alpha_a, 4) || !aligned(alpha_b, 4) || !aligned(status_dev, 4) || ldd % (out_bf16 ? 8 : 4))
    return NVFP4_ERR_ALIGN;
  nvfp4::GemmArgs a{};
  a.qa = qa;
  a.sfa = sfa;
  a.alpha_a = alpha_a;
  a.qb = qb;
  a.sfb = sfb;
  a.alpha_b = alpha_b;
  a.d = d;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldd = ldd;
  a.out_bf16 = out_bf16;
  a.status = status_dev;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = (N % 256 == 0) ? nvfp4::gemmk::launch<256, true>(a, s) : nvfp4::gemmk::launch<128, true>(a, s);
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"
