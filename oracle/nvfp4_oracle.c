/*
 * nvfp4_oracle.c -- plain, slow, obviously-correct CPU oracle for the NVFP4
 * training quantizer (E2M1 codes, one E4M3 scale per 16-element block, one
 * FP32 tensor scale).
 *
 * TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path.  Build with -O2 -ffp-contract=off and without fast-math so
 * that every float operation below is one IEEE-754 single-precision operation
 * with round-to-nearest-even, in the order written.
 *
 * Each function names the passage it follows ([P1], [P2], [SK11]; see
 * nvfp4_oracle.h).  Readings taken where the pages are silent are marked
 * "Reading:".
 */
#include "nvfp4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* [P2] Problem statement: E2M1 has steps of 0.5 on [0,2], 1 on [2,4] and 2 on
 * [4,6]; the representable magnitudes are therefore these eight, and the code
 * of a magnitude is its position in this list. */
static const float kGrid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float nvfp4ref_e2m1_value(int idx) { return kGrid[idx & 7]; }

float nvfp4ref_bf16_to_f32(uint16_t h) {
  /* bfloat16 is the upper half of a binary32; widening is exact. */
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round-to-nearest onto the E2M1 grid.  Reading: ties go to the even code
 * (the code whose mantissa bit is 0), the IEEE rule for a 1-bit mantissa.
 * m is a magnitude already clamped to the block maximum (<= 6). */
int nvfp4ref_round_rn(float m) {
  int best = 0;
  double bestd = fabs((double)m - (double)kGrid[0]);
  for (int k = 1; k < 8; ++k) {
    double dk = fabs((double)m - (double)kGrid[k]);
    if (dk < bestd || (dk == bestd && (k % 2) == 0)) {
      best = k;
      bestd = dk;
    }
  }
  return best;
}

/* [P1] section 2d: stochastic rounding rounds up with probability equal to
 * the fractional distance (1.4 -> 1 with p=0.6, -> 2 with p=0.4).
 * Reading: lo/hi are the grid neighbours of m; p = (m-lo)/(hi-lo) (exact: the
 * numerator is exact by Sterbenz and the divisor a power of two);
 * u = (word >> 8) * 2^-24 (exact); the result is hi iff u < p. */
int nvfp4ref_round_sr(float m, uint32_t word) {
  int lo = 0;
  for (int k = 0; k < 8; ++k)
    if (kGrid[k] <= m) lo = k;
  if (kGrid[lo] == m || lo == 7) return lo;
  int hi = lo + 1;
  float p = (m - kGrid[lo]) / (kGrid[hi] - kGrid[lo]);
  float u = (float)(word >> 8) * 0x1p-24f;
  return (u < p) ? hi : lo;
}

/* FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
 * finite 448, subnormal step 2^-9, no infinity) -- the block-scale format of
 * [P1] section 1 and [P2] Implementation details.  Reading: round to nearest,
 * ties to even mantissa, and values beyond 448 saturate to 448 (0x7E); the
 * input is a non-negative ratio of magnitudes. */
uint8_t nvfp4ref_e4m3_encode(float t) {
  double v = (double)t;
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  int E;
  (void)frexp(v, &E); /* v in [2^(E-1), 2^E) */
  int e = E - 1;
  if (e < -6) { /* below the smallest normal 2^-6: multiples of 2^-9 */
    double q = rint(v * 512.0); /* 0..8; 8 encodes 2^-6 (0x08) correctly */
    return (uint8_t)q;
  }
  /* 0..8; 8 carries into the exponent.  v < 448 keeps the result <= 0x7E. */
  double mant = rint((ldexp(v, -e) - 1.0) * 8.0);
  int code = ((e + 7) << 3) + (int)mant;
  return (uint8_t)code;
}

float nvfp4ref_e4m3_value(uint8_t e) {
  int ex = (e >> 3) & 0xF;
  int man = e & 7;
  if (ex == 0) return (float)ldexp((double)man, -9);
  return (float)ldexp(1.0 + (double)man / 8.0, ex - 7);
}

/* [SK11] Philox4x32 with 10 rounds.  One round multiplies counter words 0 and
 * 2 by the two published constants, swaps the halves of the products and
 * mixes in the odd counter words and the round key; the key is advanced by
 * the two Weyl constants between rounds. */
void nvfp4ref_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* [P1] section 2b: the Hadamard transform is randomised by signs.
 * Reading: one sign vector of 16 entries per call, drawn from Philox4x32-10
 * keyed by the RHT seed at counter (0,0,0,1); bit j of word 0 set means
 * sign j is -1.  Counter word 3 = 1 keeps these draws apart from the
 * stochastic-rounding draws, whose word 3 is 0. */
uint16_t nvfp4ref_rht_signs(uint64_t rht_seed) {
  uint32_t key[2] = {(uint32_t)rht_seed, (uint32_t)(rht_seed >> 32)};
  uint32_t ctr[4] = {0u, 0u, 0u, 1u};
  uint32_t out[4];
  nvfp4ref_philox4x32_10(ctr, key, out);
  return (uint16_t)(out[0] & 0xFFFFu);
}

/* Sylvester Hadamard matrix of order 16: H[i][j] = (-1)^popcount(i & j). */
int nvfp4ref_hadamard16(int i, int j) {
  int v = i & j, parity = 0;
  while (v) {
    parity ^= (v & 1);
    v >>= 1;
  }
  return parity ? -1 : 1;
}

/* [P1] section 2b: random Hadamard transform of one 16-vector,
 * y = (1/4) * H16 * (s . x), an orthonormal map.  Reading: the sum is formed
 * in double (exact for sixteen bfloat16 terms of realistic range) and rounded
 * once to float. */
void nvfp4ref_rht16(const float x[16], uint16_t signs, float y[16]) {
  for (int i = 0; i < 16; ++i) {
    double acc = 0.0;
    for (int j = 0; j < 16; ++j) {
      double sj = ((signs >> j) & 1u) ? -1.0 : 1.0;
      acc += (double)nvfp4ref_hadamard16(i, j) * sj * (double)x[j];
    }
    y[i] = (float)(0.25 * acc);
  }
}

/* Reading: the 4/6 error sums use one fixed order, a perfect binary tree over
 * the block's elements in block order (adjacent pairs first, halves last). */
float nvfp4ref_tree_sum(const float* a, int n) {
  if (n == 1) return a[0];
  float left = nvfp4ref_tree_sum(a, n / 2);
  float right = nvfp4ref_tree_sum(a + n / 2, n / 2);
  return left + right;
}

/* One block at block maximum Q ([P2] Problem statement: standard NVFP4 maps
 * the block maximum to 6; [P2] Methodology: 4/6 also tries 4).
 *   b = max|z|;  t = b / (Q*alpha);  e = E4M3(t);  d = e*alpha;
 *   v = z * (1/d);  m = min(|v|, Q);  code = sign<<3 | round(m).
 * Reading: the reciprocal is taken once per block and multiplied in; a block
 * whose scale byte rounds to zero (d == 0) keeps only the signs. */
void nvfp4ref_quant_block(const float* z, int n, float alpha, int Q, const uint32_t* words,
                          uint8_t* codes, uint8_t* e_out, float* d_out) {
  float b = 0.0f;
  for (int i = 0; i < n; ++i) b = fmaxf(b, fabsf(z[i]));
  float t = 0.0f;
  if (b > 0.0f) {
    float den = (float)Q * alpha;
    t = b / den;
  }
  uint8_t e = nvfp4ref_e4m3_encode(t);
  float d = nvfp4ref_e4m3_value(e) * alpha;
  float inv = (d != 0.0f) ? 1.0f / d : 0.0f;
  for (int i = 0; i < n; ++i) {
    int sign = signbit(z[i]) ? 1 : 0;
    int idx = 0;
    if (d != 0.0f) {
      float v = z[i] * inv;
      float m = fminf(fabsf(v), (float)Q);
      idx = words ? nvfp4ref_round_sr(m, words[i]) : nvfp4ref_round_rn(m);
    }
    codes[i] = (uint8_t)((sign << 3) | idx);
  }
  *e_out = e;
  *d_out = d;
}

/* [P2] Methodology, steps 2-3: the error of a candidate is measured against
 * the original values.  err_i = z_i - val(q_i)*d, the exact difference
 * rounded once to float (C99 fmaf).  MAE sums |err|, MSE sums err*err (the
 * square rounded to float), both over the fixed tree; MAXERR takes the
 * largest |err|.  Reading: sums stand for means (equal block sizes). */
float nvfp4ref_block_error(const float* z, int n, const uint8_t* codes, float d, int sel) {
  float terms[256];
  float mx = 0.0f;
  for (int i = 0; i < n; ++i) {
    float val = kGrid[codes[i] & 7];
    if (codes[i] & 8) val = -val;
    float err = fmaf(-val, d, z[i]);
    if (sel == REF_SEL_MSE) {
      terms[i] = err * err;
    } else {
      terms[i] = fabsf(err);
    }
    mx = fmaxf(mx, fabsf(err));
  }
  if (sel == REF_SEL_MAXERR) return mx;
  return nvfp4ref_tree_sum(terms, n);
}

/* ------------------------------------------------------------------------ */

static int flags_valid(uint32_t flags, int sel) {
  uint32_t known = REF_ROWWISE | REF_COLWISE | REF_2D | REF_RHT_ROW | REF_RHT_COL | REF_SR | REF_46;
  if (flags & ~known) return 0;
  if (!(flags & (REF_ROWWISE | REF_COLWISE))) return 0;
  if ((flags & REF_2D) && (flags & (REF_RHT_ROW | REF_RHT_COL))) return 0;
  if ((flags & REF_RHT_ROW) && !(flags & REF_ROWWISE)) return 0;
  if ((flags & REF_RHT_COL) && !(flags & REF_COLWISE)) return 0;
  if ((flags & REF_46) && (sel < REF_SEL_MAE || sel > REF_SEL_MAXERR)) return 0;
  return 1;
}

static int shape_valid(int64_t M, int64_t N, int64_t ld, uint32_t flags) {
  if (M < 0 || N < 0) return REF_ERR_SHAPE;
  if (N % 16) return REF_ERR_SHAPE;
  if ((flags & (REF_COLWISE | REF_2D)) && (M % 16)) return REF_ERR_SHAPE;
  if (ld < N) return REF_ERR_SHAPE;
  if (ld % 8) return REF_ERR_ALIGN;
  return REF_OK;
}

static void row_vector(const uint16_t* x, int64_t ld, int64_t r, int64_t c0, float z[16]) {
  for (int j = 0; j < 16; ++j) z[j] = nvfp4ref_bf16_to_f32(x[r * ld + c0 + j]);
}

static void col_vector(const uint16_t* x, int64_t ld, int64_t r0, int64_t c, float z[16]) {
  for (int j = 0; j < 16; ++j) z[j] = nvfp4ref_bf16_to_f32(x[(r0 + j) * ld + c]);
}

/* [P2] Implementation details: the tensor scale is taken from the tensor's
 * largest magnitude.  amax[0] belongs to the rowwise copy, amax[1] to the
 * columnwise copy; a copy that is Hadamard-transformed takes the largest
 * magnitude of its transformed values (Reading: the scale must cover what is
 * actually quantized). */
/* max of magnitudes that keeps a NaN once one has been seen */
static float max_keep_nan(float acc, float a) {
  if (isnan(acc)) return acc;
  if (isnan(a)) return a;
  return (a > acc) ? a : acc;
}

int nvfp4ref_amax(const uint16_t* x, int64_t M, int64_t N, int64_t ld, uint32_t flags,
                  uint64_t rht_seed, float amax[2]) {
  if (!amax || (!x && M > 0 && N > 0)) return REF_ERR_NULL;
  if (!flags_valid(flags, REF_SEL_MAE)) return REF_ERR_FLAGS;
  int st = shape_valid(M, N, ld, flags);
  if (st != REF_OK) return st;
  uint16_t signs = nvfp4ref_rht_signs(rht_seed);
  float plain = 0.0f, z[16], y[16];
  for (int64_t r = 0; r < M; ++r)
    for (int64_t c = 0; c < N; ++c) plain = max_keep_nan(plain, fabsf(nvfp4ref_bf16_to_f32(x[r * ld + c])));
  amax[0] = plain;
  amax[1] = plain;
  if (flags & REF_RHT_ROW) {
    float m = 0.0f;
    for (int64_t r = 0; r < M; ++r)
      for (int64_t c0 = 0; c0 < N; c0 += 16) {
        row_vector(x, ld, r, c0, z);
        nvfp4ref_rht16(z, signs, y);
        for (int j = 0; j < 16; ++j) m = max_keep_nan(m, fabsf(y[j]));
      }
    amax[0] = m;
  }
  if (flags & REF_RHT_COL) {
    float m = 0.0f;
    for (int64_t r0 = 0; r0 < M; r0 += 16)
      for (int64_t c = 0; c < N; ++c) {
        col_vector(x, ld, r0, c, z);
        nvfp4ref_rht16(z, signs, y);
        for (int j = 0; j < 16; ++j) m = max_keep_nan(m, fabsf(y[j]));
      }
    amax[1] = m;
  }
  return REF_OK;
}

/* Philox words for element (r, c) of the source tensor: counter = element
 * index (the counter_offset plus the element's row-major index in the
 * source tensor), key = seed. */
static void element_words(uint64_t sr_seed, uint64_t counter_offset, int64_t N, int64_t r, int64_t c,
                          uint32_t out[4]) {
  uint64_t i = counter_offset + (uint64_t)r * (uint64_t)N + (uint64_t)c;
  uint32_t ctr[4] = {(uint32_t)i, (uint32_t)(i >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)sr_seed, (uint32_t)(sr_seed >> 32)};
  nvfp4ref_philox4x32_10(ctr, key, out);
}

/* One block, standard or 4/6.  [P2] Methodology: with 4/6 the block is
 * quantized at maximum 6 and at maximum 4, the error of each is measured and
 * the lower one kept.  Reading: 4 is kept only if its score is strictly lower
 * (ties keep the standard 6). */
static uint8_t quantize_one_block(const float* z, int n, float alpha, int use46, int sel,
                                  const uint32_t* words, uint8_t* codes) {
  uint8_t e6, e4;
  float d6, d4;
  nvfp4ref_quant_block(z, n, alpha, 6, words, codes, &e6, &d6);
  if (!use46) return e6;
  uint8_t codes4[256];
  nvfp4ref_quant_block(z, n, alpha, 4, words, codes4, &e4, &d4);
  float s6 = nvfp4ref_block_error(z, n, codes, d6, sel);
  float s4 = nvfp4ref_block_error(z, n, codes4, d4, sel);
  if (s4 < s6) {
    memcpy(codes, codes4, (size_t)n);
    return e4;
  }
  return e6;
}

static void put_code(uint8_t* q, int64_t row_bytes, int64_t r, int64_t c, uint8_t code) {
  uint8_t* p = &q[r * row_bytes + c / 2];
  if (c % 2 == 0)
    *p = (uint8_t)((*p & 0xF0) | (code & 0x0F));
  else
    *p = (uint8_t)((*p & 0x0F) | ((code & 0x0F) << 4));
}

static int check_scale(float A) {
  if (!isfinite(A)) return REF_ERR_NONFINITE;
  if (A > 0.0f && A < 0x1p-100f) return REF_ERR_RANGE;
  return REF_OK;
}

int nvfp4ref_quantize_rows(const uint16_t* x, int64_t M, int64_t N, int64_t ld,
                           const float amax[2], uint32_t flags, int sel, uint64_t sr_seed,
                           uint64_t rht_seed, uint64_t counter_offset, int64_t row0,
                           int64_t row1, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                           uint8_t* s_col, float alpha[2]) {
  if (!amax || !alpha) return REF_ERR_NULL;
  if (!flags_valid(flags, sel)) return REF_ERR_FLAGS;
  int st = shape_valid(M, N, ld, flags);
  if (st != REF_OK) return st;
  int do_row = (flags & REF_ROWWISE) != 0, do_col = (flags & REF_COLWISE) != 0;
  if (M > 0 && N > 0) {
    if (!x) return REF_ERR_NULL;
    if (do_row && (!q_row || !s_row)) return REF_ERR_NULL;
    if (do_col && (!q_col || !s_col)) return REF_ERR_NULL;
  }
  if (row0 < 0 || row1 > M || row0 > row1 || row0 % 16 || (row1 % 16 && row1 != M))
    return REF_ERR_SHAPE;
  int use46 = (flags & REF_46) != 0;
  int use_sr = (flags & REF_SR) != 0;
  /* [P2] Implementation details: alpha = amax / (6*448), or amax / (6*256)
   * with 4/6 so that the 1.5x larger max-4 scale stays inside E4M3. */
  float denom = use46 ? 1536.0f : 2688.0f;
  alpha[0] = amax[0] / denom;
  alpha[1] = amax[1] / denom;
  if (do_row || (flags & REF_2D)) {
    st = check_scale(amax[0]);
    if (st != REF_OK) return st;
  }
  if (do_col) {
    st = check_scale(amax[1]);
    if (st != REF_OK) return st;
  }
  uint16_t signs = nvfp4ref_rht_signs(rht_seed);
  float z[256], y[16];
  uint8_t codes[256];
  uint32_t words[256], w4[4];

  if (flags & REF_2D) {
    /* [P1] section 2c: one scale per 16x16 tile, shared by the rowwise and
     * the transposed copy, so both copies hold the same quantized weight.
     * Both copies use Philox word 0 so that their codes stay transposes. */
    for (int64_t tr = row0; tr < row1; tr += 16)
      for (int64_t tc = 0; tc < N; tc += 16) {
        for (int k = 0; k < 256; ++k) {
          int64_t r = tr + k / 16, c = tc + k % 16;
          z[k] = nvfp4ref_bf16_to_f32(x[r * ld + c]);
          if (use_sr) {
            element_words(sr_seed, counter_offset, N, r, c, w4);
            words[k] = w4[0];
          }
        }
        uint8_t e = quantize_one_block(z, 256, alpha[0], use46, sel, use_sr ? words : NULL, codes);
        for (int k = 0; k < 256; ++k) {
          int64_t r = tr + k / 16, c = tc + k % 16;
          if (do_row) put_code(q_row, N / 2, r, c, codes[k]);
          if (do_col) put_code(q_col, M / 2, c, r, codes[k]);
        }
        for (int k = 0; k < 16; ++k) {
          if (do_row) s_row[(tr + k) * (N / 16) + tc / 16] = e;
          if (do_col) s_col[(tc + k) * (M / 16) + tr / 16] = e;
        }
      }
    return REF_OK;
  }

  if (do_row) {
    for (int64_t r = row0; r < row1; ++r)
      for (int64_t c0 = 0; c0 < N; c0 += 16) {
        row_vector(x, ld, r, c0, z);
        if (flags & REF_RHT_ROW) {
          nvfp4ref_rht16(z, signs, y);
          memcpy(z, y, sizeof y);
        }
        if (use_sr)
          for (int j = 0; j < 16; ++j) {
            element_words(sr_seed, counter_offset, N, r, c0 + j, w4);
            words[j] = w4[0]; /* rowwise copy: word 0 */
          }
        uint8_t e = quantize_one_block(z, 16, alpha[0], use46, sel, use_sr ? words : NULL, codes);
        for (int j = 0; j < 16; ++j) put_code(q_row, N / 2, r, c0 + j, codes[j]);
        s_row[r * (N / 16) + c0 / 16] = e;
      }
  }
  if (do_col) {
    for (int64_t r0 = row0; r0 < row1; r0 += 16)
      for (int64_t c = 0; c < N; ++c) {
        col_vector(x, ld, r0, c, z);
        if (flags & REF_RHT_COL) {
          nvfp4ref_rht16(z, signs, y);
          memcpy(z, y, sizeof y);
        }
        if (use_sr)
          for (int j = 0; j < 16; ++j) {
            element_words(sr_seed, counter_offset, N, r0 + j, c, w4);
            words[j] = w4[1]; /* columnwise copy: word 1 */
          }
        uint8_t e = quantize_one_block(z, 16, alpha[1], use46, sel, use_sr ? words : NULL, codes);
        for (int j = 0; j < 16; ++j) put_code(q_col, M / 2, c, r0 + j, codes[j]);
        s_col[c * (M / 16) + r0 / 16] = e;
      }
  }
  return REF_OK;
}

int nvfp4ref_quantize(const uint16_t* x, int64_t M, int64_t N, int64_t ld, const float amax[2],
                      uint32_t flags, int sel, uint64_t sr_seed, uint64_t rht_seed,
                      uint64_t counter_offset, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                      uint8_t* s_col, float alpha[2]) {
  return nvfp4ref_quantize_rows(x, M, N, ld, amax, flags, sel, sr_seed, rht_seed, counter_offset,
                                0, M, q_row, s_row, q_col, s_col, alpha);
}

/* fp32 -> bfloat16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* Dequantize: x^ = val(q) * (e * alpha), the reconstruction that the 4/6
 * error of [P2] Methodology is measured against.  out is float (out_is_bf16
 * = 0) or bfloat16 bits rounded to nearest even (out_is_bf16 = 1). */
int nvfp4ref_dequantize(const uint8_t* q, const uint8_t* s, float alpha, int64_t rows,
                        int64_t cols, int out_is_bf16, void* out) {
  if (rows < 0 || cols < 0 || cols % 16) return REF_ERR_SHAPE;
  if (rows > 0 && cols > 0 && (!q || !s || !out)) return REF_ERR_NULL;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = q[r * (cols / 2) + c / 2];
      uint8_t code = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
      float d = nvfp4ref_e4m3_value(s[r * (cols / 16) + c / 16]) * alpha;
      float val = kGrid[code & 7];
      if (code & 8) val = -val;
      float xh = val * d;
      if (out_is_bf16)
        ((uint16_t*)out)[r * cols + c] = f32_to_bf16_rne(xh);
      else
        ((float*)out)[r * cols + c] = xh;
    }
  return REF_OK;
}

/* Error histogram of a rowwise copy over the scaled value ("Four Over Six
 * (4/6)" technical summary, Problem statement: values between 4 and 6 at
 * block scale 6 -- around scaled value 5 -- carry the rounding error that
 * matters).  For every element of every block with a nonzero maximum b:
 * v = (6|x|)/b, bin = min(floor((v*nbins)/6), nbins-1); e = (6|x - x^|)/b with
 * x^ = val(q) * (e4m3(s) * alpha) as the dequantizer forms it; the bin adds 1
 * to hist[bin], trunc(e * 2^24) to hist[nbins + bin] and trunc(e*e * 2^32) to
 * hist[2*nbins + bin].  Each step is one float operation, in that order. */
int nvfp4ref_error_histogram(const uint16_t* x, int64_t M, int64_t N, int64_t ld, const uint8_t* q,
                             const uint8_t* s, float alpha, int nbins, uint64_t* hist) {
  if (M < 0 || N < 0 || N % 16 || ld < N || nbins < 1 || nbins > 1024) return REF_ERR_SHAPE;
  for (int64_t r = 0; r < M; ++r)
    for (int64_t c0 = 0; c0 < N; c0 += 16) {
      float b = 0.0f;
      for (int j = 0; j < 16; ++j) {
        float a = fabsf(nvfp4ref_bf16_to_f32(x[r * ld + c0 + j]));
        if (a > b) b = a;
      }
      if (!(b > 0.0f)) continue;
      float d = nvfp4ref_e4m3_value(s[r * (N / 16) + c0 / 16]) * alpha;
      for (int j = 0; j < 16; ++j) {
        int64_t c = c0 + j;
        float xv = nvfp4ref_bf16_to_f32(x[r * ld + c]);
        uint8_t byte = q[r * (N / 2) + c / 2];
        uint8_t code = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
        float val = kGrid[code & 7];
        if (code & 8) val = -val;
        float xh = val * d;
        float six_x = 6.0f * fabsf(xv);
        float v = six_x / b;
        float scaled = v * (float)nbins;
        int bin = (int)floorf(scaled / 6.0f);
        if (bin > nbins - 1) bin = nbins - 1;
        float diff = xv - xh;
        float six_e = 6.0f * fabsf(diff);
        float e = six_e / b;
        float e24 = e * 0x1p24f;
        float ee = e * e;
        float ee32 = ee * 0x1p32f;
        hist[bin] += 1u;
        hist[nbins + bin] += (uint64_t)e24;
        hist[2 * nbins + bin] += (uint64_t)ee32;
      }
    }
  return REF_OK;
}

/* NVFP4 GEMM of two operands in the layout the quantizer writes ("NVFP4
 * revolutionizes AI training" headline page: Blackwell computes matrix
 * products (GEMM) on FP4 operands natively).  A is M x K, B is N x K, both
 * with 16-element blocks along K (codes M x K/2 and N x K/2 bytes, plain
 * scales M x K/16 and N x K/16); D = A * B^T, M x N floats.
 * Reading: each operand is dequantized exactly as nvfp4ref_dequantize forms
 * it (x^ = val(q) * (e4m3(s) * alpha), rounded to float), the products and
 * their sum over k are formed in double, and each element is rounded once to
 * float. */
int nvfp4ref_gemm(const uint8_t* qa, const uint8_t* sa, float alpha_a, const uint8_t* qb,
                  const uint8_t* sb, float alpha_b, int64_t M, int64_t N, int64_t K, float* d) {
  if (M < 0 || N < 0 || K < 0 || K % 16) return REF_ERR_SHAPE;
  if (M == 0 || N == 0) return REF_OK;
  if (!d || (K > 0 && (!qa || !sa || !qb || !sb))) return REF_ERR_NULL;
  float* xa = (float*)malloc(sizeof(float) * (size_t)(M * (K > 0 ? K : 1)));
  float* xb = (float*)malloc(sizeof(float) * (size_t)(N * (K > 0 ? K : 1)));
  if (!xa || !xb) {
    free(xa);
    free(xb);
    return REF_ERR_NULL;
  }
  if (K > 0) {
    nvfp4ref_dequantize(qa, sa, alpha_a, M, K, 0, xa);
    nvfp4ref_dequantize(qb, sb, alpha_b, N, K, 0, xb);
  }
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += (double)xa[m * K + k] * (double)xb[n * K + k];
      d[m * N + n] = (float)acc;
    }
  free(xa);
  free(xb);
  return REF_OK;
}
