// nvfp4_device.cuh -- device building blocks of the NVFP4 quantizer (sm_103a).
//
// Every floating-point step of the quantizer's contract is written with an
// explicit round-to-nearest intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn,
// __frcp_rn, __fmaf_rn) so that the compiler can neither fuse nor reorder it;
// the library is also built with -fmad=false.  The E2M1 and E4M3 conversions
// use the Blackwell cvt instructions (the "cvt family" that the 4/6 page's
// Implementation details name), written here as inline PTX.
//
// Sources: "Four Over Six (4/6)" technical summary (Problem statement:
// E2M1 steps and [-6,6] block scaling; Methodology: dual quantization, error,
// selection; Implementation details: alpha over 256), "Pretraining Large
// Language Models with NVFP4" sections 2b-2d (RHT, 2D scaling, stochastic
// rounding), Salmon et al. SC'11 (Philox4x32-10).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace nvfp4 {

constexpr float kAlphaDen = 2688.0f;    // 6 * 448: block max 6, E4M3 max 448
constexpr float kAlphaDen46 = 1536.0f;  // 6 * 256: headroom for the 1.5x max-4 scale
constexpr float kMinAmax = 0x1p-100f;   // below this the per-block reciprocal may overflow

// status values written to the device status word (same integers as nvfp4.h)
constexpr int kStatusNonFinite = -6;
constexpr int kStatusRange = -7;
constexpr int kStatusPipeline = -8;

// ---------------------------------------------------------------- bf16
// Exact widening of the low / high bf16 half of a word by bit placement
// (integer pipe).
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The same widening as a mixed-precision add of -0.0 (exact, keeps the sign
// of zero) so that it runs on the floating-point pipe, which has twice the
// integer pipe's throughput.
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t v) {
  float2 r;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.bf16 %0, l, 0f80000000;\n"
      " add.rn.f32.bf16 %1, h, 0f80000000;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(v));
  return r;
}
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t v) {
  float2 r;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.f16 %0, l, 0f80000000;\n"
      " add.rn.f32.f16 %1, h, 0f80000000;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(v));
  return r;
}

// Packed FP32 pairs (Blackwell f32x2): two IEEE round-to-nearest operations
// per instruction, each rounded exactly like its scalar counterpart.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rc, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rr, ra, rb, rc;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " sub.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// max(|a|, |b|) per bf16 half (the sign of the result is meaningless; mask it)
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest magnitude of the 16 bf16 values in w[0..7], as float (exact).
__device__ __forceinline__ float block_absmax16(const uint32_t* w) {
  const uint32_t a = absmax_bf16x2(absmax_bf16x2(w[0], w[1]), absmax_bf16x2(w[2], w[3]));
  const uint32_t b = absmax_bf16x2(absmax_bf16x2(w[4], w[5]), absmax_bf16x2(w[6], w[7]));
  const uint32_t m = absmax_bf16x2(a, b) & 0x7FFF7FFFu;
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------- E4M3 scale
// Scale byte of a non-negative ratio: round to nearest even, saturate at 448.
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

// Value of a scale byte (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float e4m3_value(uint32_t e) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)e));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// ---------------------------------------------------------------- E2M1 codes
// Two values -> one byte of codes (first value in the low nibble), round to
// nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t e2m1x2(float first, float second) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}"
      : "=r"(r)
      : "f"(second), "f"(first));
  return r;
}

// Eight values -> eight nibbles (value j in bits 4j..4j+3).
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Signed grid values of the two codes in the low byte of `byte2` (exact).
__device__ __forceinline__ float2 e2m1x2_values(uint32_t byte2) {
  uint32_t h2;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "r"(byte2));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon et al., SC'11.  Counter (c0, c1, 0, 0), key (k0, k1); returns words
// 0 and 1 of the output block.
__device__ __forceinline__ uint2 philox_w01(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t c2 = 0u, c3 = 0u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint2(c0, c1);
}

// The same words for a counter (lo, hi, 0, 0) whose second-round product of
// word 0, M0 * (hi ^ k0), is given: in the first round word 2 is zero, so
// word 0 leaves it as hi ^ k0 and word 1 as zero, and that product depends
// on the high word and the key alone -- counters that share a high word
// share it.
__device__ __forceinline__ uint2 philox_w01_shared_hi(uint32_t lo, uint64_t p0_round1, uint32_t k0, uint32_t k1) {
  const uint64_t q = (uint64_t)0xD2511F53u * lo;  // round 0
  uint32_t c2 = (uint32_t)(q >> 32) ^ k1;
  uint32_t c3 = (uint32_t)q;
  k0 += 0x9E3779B9u;
  k1 += 0xBB67AE85u;
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;  // round 1
  uint32_t c0 = (uint32_t)(p1 >> 32) ^ k0;
  uint32_t c1 = (uint32_t)p1;
  c2 = (uint32_t)(p0_round1 >> 32) ^ c3 ^ k1;
  c3 = (uint32_t)p0_round1;
  k0 += 0x9E3779B9u;
  k1 += 0xBB67AE85u;
#pragma unroll
  for (int round = 2; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1r = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1r >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1r;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint2(c0, c1);
}

// Words 0 and 1 of the NC counters base + j * stride, j = 0..NC-1
// (stride < 2^32).  When all of them share their high word -- every group but
// one that crosses a multiple of 2^32 -- the second-round product of word 0 is
// formed once for the group.
template <int NC, bool W1>
__device__ __forceinline__ void philox_group_w01(uint64_t base, uint32_t stride, uint32_t k0, uint32_t k1,
                                                 uint32_t* w0, uint32_t* w1) {
  const uint64_t last = base + (uint64_t)(NC - 1) * stride;
  if ((uint32_t)(base >> 32) == (uint32_t)(last >> 32)) {
    const uint64_t p0r1 = (uint64_t)0xD2511F53u * ((uint32_t)(base >> 32) ^ k0);
    const uint32_t lo = (uint32_t)base;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const uint2 r = philox_w01_shared_hi(lo + (uint32_t)j * stride, p0r1, k0, k1);
      w0[j] = r.x;
      if (W1) w1[j] = r.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const uint64_t i = base + (uint64_t)j * stride;
      const uint2 r = philox_w01((uint32_t)i, (uint32_t)(i >> 32), k0, k1);
      w0[j] = r.x;
      if (W1) w1[j] = r.y;
    }
  }
}

// RHT sign bits: word 0 of Philox(key = seed, counter = (0,0,0,1)).
__device__ __forceinline__ uint32_t rht_sign_bits(uint32_t k0, uint32_t k1) {
  uint32_t c0 = 0u, c1 = 0u, c2 = 0u, c3 = 1u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0 & 0xFFFFu;
}

// ---------------------------------------------------------------- rounding
// Stochastic rounding of v onto the E2M1 grid with block maximum Q: with
// m = min(|v|, Q) between grid neighbours lo <= m < hi, return hi iff
// u = (w >> 8) * 2^-24 < p = (m - lo) / (hi - lo); the sign of v is kept.
// The step hi - lo is 2^(e-1) for m in [2^e, 2^(e+1)), e = 0, 1, 2, and 1/2
// below 1 (max(2^e, 1) / 2, formed on the exponent field, as is its
// reciprocal).  In units of the step m is t = f + p with f = floor(t) the
// grid point lo, and hi is chosen exactly when t - u > f; since u lies in
// [0, 1), t - u lies in (f, f + 1) when u < p and in (f - 1, f] otherwise,
// so the grid point is q = ceil(t - u).  t - u is formed by one fused
// multiply-add rounded upward: that rounding never passes an integer (the
// integers up to 4 are floats), so ceil sees the exact decision.
__device__ __forceinline__ float sr_round(float v, float Q, uint32_t w) {
  const float m = fminf(fabsf(v), Q);
  const int sb = max((int)(__float_as_uint(m) & 0x7F800000u) - 0x00800000, 0x3F000000);
  const float step = __int_as_float(sb);
  const float rstep = __int_as_float(0x7F000000 - sb);
  const float t = __fmul_rn(m, rstep);  // exact: a power-of-two scaling
  const float d = __fmaf_ru(__uint2float_rn(w >> 8), -0x1p-24f, t);
  const float g = __fmul_rn(ceilf(d), step);
  return copysignf(g, v);
}

// ---------------------------------------------------------------- block scale
struct BlockScale {
  uint32_t e;  // E4M3 byte
  float d;     // e * alpha
  float inv;   // 1 / d (0 when d == 0: every code becomes a signed zero)
};

// b = block max, Q = 6 or 4:  t = b / (Q*alpha), e = E4M3(t), d = e*alpha.
__device__ __forceinline__ BlockScale block_scale(float b, float alpha, float Q) {
  BlockScale s;
  const float den = __fmul_rn(Q, alpha);
  const float t = (b > 0.0f) ? __fdiv_rn(b, den) : 0.0f;
  s.e = e4m3_encode(t);
  s.d = __fmul_rn(e4m3_value(s.e), alpha);
  s.inv = (s.d != 0.0f) ? __frcp_rn(s.d) : 0.0f;
  return s;
}

// The quotient b / den for the scale byte, from rden = fl(1/den) without a
// division: q0 = fl(b * rden) is within 2 ulp of b / den, and one residual
// correction q1 = q0 + (b - q0*den) * rden (two fused multiply-adds; the
// residual of a close quotient is exact) brings it within an ulp of
// fl(b / den).  That is not always fl(b / den) itself, but its E4M3 byte is
// the byte of fl(b / den) for every pair of a finite bf16 block maximum and an
// accepted bf16 amax, for fp32 amax values between them and for random fp32
// maxima -- checked exhaustively on the device by the test-only self-check
// library (tests/selftest); the bare product gets tens of thousands of those
// bytes wrong.
// b >= 0 finite, den > 0 normal, or den == rden == 0 with b == 0.
__device__ __forceinline__ float quotient_rn(float b, float den, float rden) {
  const float q = __fmul_rn(b, rden);
  return __fmaf_rn(__fmaf_rn(-q, den, b), rden, q);
}

// Scale byte of a block: e = E4M3(fl(b / den)), den = Q * alpha.  Every
// quotient from 464 up saturates to 448 (byte 0x7E); the cap keeps the
// corrections from turning an overflowing quotient (b >> amax, possible with a
// caller-supplied amax) into NaN, whose byte would be 0x7F.
__device__ __forceinline__ uint32_t scale_byte(float b, float den, float rden) {
  return e4m3_encode(fminf(quotient_rn(b, den, rden), 1.0e6f));  // b == 0 gives byte 0
}

// A max-4 candidate needs its scaled values clamped to +-4 before rounding to
// nearest only when its scale byte is subnormal (< 8: E4M3 rounding error up
// to 50 %) or saturated (0x7E: the block maximum may exceed 448 * 4 * alpha,
// e.g. with a caller-supplied amax); otherwise every scaled value is at most
// 4.25 and rounds to at most 4.
__device__ __forceinline__ bool max4_needs_clamp(uint32_t e) { return e < 8u || e >= 0x7Eu; }

// Per-copy table of d = e*alpha and 1/d for every scale byte e (0..127),
// filled once per CTA: entry e = (d, inv) exactly as block_scale computes them.
__device__ __forceinline__ float2 scale_entry(uint32_t e, float alpha) {
  const float d = __fmul_rn(e4m3_value(e), alpha);
  return make_float2(d, (d != 0.0f) ? __frcp_rn(d) : 0.0f);
}

// Two values -> one code byte, plus the two codes' signed grid values as an
// f16x2 (low half = first value).
__device__ __forceinline__ uint32_t e2m1x2_enc_dec(float first, float second, uint32_t& h2) {
  uint32_t byte;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n cvt.rn.f16x2.e2m1x2 %1, t;\n"
      " cvt.u32.u8 %0, t;\n}"
      : "=r"(byte), "=r"(h2)
      : "f"(second), "f"(first));
  return byte;
}

// Eight values -> eight nibbles (value j in bits 4j..4j+3), plus the codes'
// signed grid values as four f16x2 words (h[k] holds values 2k, 2k+1).
__device__ __forceinline__ uint32_t e2m1x8_enc_dec(const float* v, uint32_t* h) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %4, b3;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Four bytes (low byte of each argument) -> one word, first argument lowest.
__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// ---------------------------------------------------------------- 4/6 error terms
enum Sel : int { kSelMAE = 0, kSelMSE = 1, kSelMax = 2 };

// Error term of one element: err = z - val*d rounded once (fma), then |err|
// (MAE, MAX) or err*err (MSE).
__device__ __forceinline__ float err_term(float z, float val, float d, int sel) {
  const float err = __fmaf_rn(-val, d, z);
  return (sel == kSelMSE) ? __fmul_rn(err, err) : fabsf(err);
}

// Combine two partial scores: a sum for MAE/MSE, a max for MAXERR.
__device__ __forceinline__ float err_combine(float a, float b, int sel) {
  return (sel == kSelMax) ? fmaxf(a, b) : __fadd_rn(a, b);
}

// Score of 8 consecutive elements whose codes are the 8 nibbles of `codes`,
// summed as a perfect binary tree (adjacent pairs first).
__device__ __forceinline__ float score8(const float* z, uint32_t codes, float d, int sel) {
  float t[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 val = e2m1x2_values((codes >> (8 * j)) & 0xFFu);
    t[2 * j] = err_term(z[2 * j], val.x, d, sel);
    t[2 * j + 1] = err_term(z[2 * j + 1], val.y, d, sel);
  }
  const float a = err_combine(err_combine(t[0], t[1], sel), err_combine(t[2], t[3], sel), sel);
  const float b = err_combine(err_combine(t[4], t[5], sel), err_combine(t[6], t[7], sel), sel);
  return err_combine(a, b, sel);
}

// ---------------------------------------------------------------- Hadamard
// 16-point random Hadamard transform y = (1/4) H16 (s . z), H16 in Sylvester
// order (the iterative butterfly yields natural order), s_j = -1 where bit j
// of `signs` is set.  The sign flips are exact, so they are applied to the
// packed bf16 words before widening: an XOR with a mask built from the sign
// bits (uniform across the kernel, so the masks live in uniform registers).
// A columnwise word holds row j of two neighbouring columns, a rowwise word
// elements 2j and 2j+1 of one vector.
__device__ __forceinline__ uint32_t rht_mask_col(uint32_t signs, int j) { return ((signs >> j) & 1u) * 0x80008000u; }
__device__ __forceinline__ uint32_t rht_mask_row(uint32_t signs, int j) {
  return (((signs >> (2 * j)) & 1u) << 15) | (((signs >> (2 * j + 1)) & 1u) << 31);
}

// Unnormalised butterfly on two vectors at once, held as pairs z[i] =
// (element i of the first vector, element i of the second): four stages of
// packed adds and subtracts, each rounded as its scalar counterpart.
__device__ __forceinline__ void wht16_x2(float2* z) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float2 a = z[i], b = z[i + h];
        z[i] = add2(a, b);
        z[i + h] = sub2(a, b);
      }
    }
  }
}

// Unnormalised butterfly on one vector z[0..15]: the first stage pairs
// neighbours (scalar), the later stages pair (i, i+1) with (i+h, i+h+1)
// (packed).  Same operations in the same order as the plain butterfly.
__device__ __forceinline__ void wht16(float* z) {
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float a = z[i], b = z[i + 1];
    z[i] = __fadd_rn(a, b);
    z[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      if ((i & h) == 0) {
        const float2 a = make_float2(z[i], z[i + 1]), b = make_float2(z[i + h], z[i + h + 1]);
        const float2 s = add2(a, b), d = sub2(a, b);
        z[i] = s.x;
        z[i + 1] = s.y;
        z[i + h] = d.x;
        z[i + h + 1] = d.y;
      }
    }
  }
}

// Status of a tensor amax: 0 if usable, else the status value.
__device__ __forceinline__ int amax_status(float A) {
  if (!(A <= 3.402823466e38f)) return kStatusNonFinite;  // Inf or NaN
  if (A > 0.0f && A < kMinAmax) return kStatusRange;
  return 0;
}

}  // namespace nvfp4
