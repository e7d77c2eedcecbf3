/*
 * nvfp4_oracle.h -- plain, slow CPU oracle for the NVFP4 training quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant generator with the
 * CUDA library; the flag and status values below are written out again here
 * because they are an interface (both sides must agree on what the integers
 * mean), not shared code.
 *
 * Sources (the pages the method is taken from):
 *   [P1] "Pretraining Large Language Models with NVFP4" (gist.science summary
 *        of arXiv 2509.25149): section 1 (16-element blocks, E4M3 scales),
 *        section 2b (random Hadamard transform, backward only), 2c (2D block
 *        scaling), 2d (stochastic rounding).
 *   [P2] "Four Over Six (4/6)" technical summary (gist.science, arXiv
 *        2512.02010): "Problem statement" (E2M1 steps, [-6,6] block scaling,
 *        the 66.6% gap), "Methodology" (dual quantization, error, the three
 *        selection rules), "Implementation details" (tensor scale over 256
 *        instead of 448).
 *   [SK11] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *        1, 2, 3", SC'11 -- the Philox4x32-10 generator.
 * Where the pages leave a step open, the reading taken is stated beside the
 * function that implements it.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* flags (interface values) */
#define REF_ROWWISE 1u
#define REF_COLWISE 2u
#define REF_2D 4u
#define REF_RHT_ROW 8u
#define REF_RHT_COL 16u
#define REF_SR 32u
#define REF_46 64u

/* 4/6 selection rules */
#define REF_SEL_MAE 0
#define REF_SEL_MSE 1
#define REF_SEL_MAXERR 2

/* status values */
#define REF_OK 0
#define REF_ERR_NULL (-1)
#define REF_ERR_SHAPE (-2)
#define REF_ERR_ALIGN (-3)
#define REF_ERR_FLAGS (-4)
#define REF_ERR_NONFINITE (-6)
#define REF_ERR_RANGE (-7)

/* ---- scalar building blocks (exported so the pins can test each one) ---- */
float nvfp4ref_bf16_to_f32(uint16_t h);
float nvfp4ref_e2m1_value(int idx);                 /* idx 0..7 -> grid magnitude   */
int nvfp4ref_round_rn(float m);                     /* m in [0,6] -> grid index     */
int nvfp4ref_round_sr(float m, uint32_t word);      /* m in [0,6] -> grid index     */
uint8_t nvfp4ref_e4m3_encode(float t);              /* t >= 0 -> E4M3 byte          */
float nvfp4ref_e4m3_value(uint8_t e);               /* E4M3 byte -> value           */
void nvfp4ref_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
uint16_t nvfp4ref_rht_signs(uint64_t rht_seed);     /* bit j set -> sign j is -1    */
int nvfp4ref_hadamard16(int i, int j);              /* +1 / -1                      */
void nvfp4ref_rht16(const float x[16], uint16_t signs, float y[16]);
float nvfp4ref_tree_sum(const float* a, int n);     /* n a power of two            */

/* One block of n (16 or 256) values z at tensor scale alpha and block maximum Q
 * (6 or 4).  words[] (n entries) are the SR random words, or NULL for RN.
 * Writes n codes (sign<<3 | index), the scale byte and d = e*alpha. */
void nvfp4ref_quant_block(const float* z, int n, float alpha, int Q, const uint32_t* words,
                          uint8_t* codes, uint8_t* e_out, float* d_out);
/* Error score of a block quantized with (codes, d) against z under a rule. */
float nvfp4ref_block_error(const float* z, int n, const uint8_t* codes, float d, int sel);

/* ---- whole-tensor calls (host buffers; same argument meaning as the library) ---- */
int nvfp4ref_amax(const uint16_t* x, int64_t M, int64_t N, int64_t ld, uint32_t flags,
                  uint64_t rht_seed, float amax[2]);

/* Quantize rows [row0, row1) of X (row0, row1 multiples of 16; the full tensor
 * is row0=0, row1=M).  The outputs are the FULL-size buffers; only the parts
 * that belong to those rows are written.  amax[2] comes from nvfp4ref_amax. */
int nvfp4ref_quantize_rows(const uint16_t* x, int64_t M, int64_t N, int64_t ld,
                           const float amax[2], uint32_t flags, int sel, uint64_t sr_seed,
                           uint64_t rht_seed, uint64_t counter_offset, int64_t row0,
                           int64_t row1, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                           uint8_t* s_col, float alpha[2]);

int nvfp4ref_quantize(const uint16_t* x, int64_t M, int64_t N, int64_t ld, const float amax[2],
                      uint32_t flags, int sel, uint64_t sr_seed, uint64_t rht_seed,
                      uint64_t counter_offset, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                      uint8_t* s_col, float alpha[2]);

/* codes (rows x cols/2 bytes) + scales (rows x cols/16) + alpha -> float
 * values (out_is_bf16 = 0) or bfloat16 bits (out_is_bf16 = 1) */
int nvfp4ref_dequantize(const uint8_t* q, const uint8_t* s, float alpha, int64_t rows,
                        int64_t cols, int out_is_bf16, void* out);

/* D = A * B^T of two NVFP4 operands (A: M x K, B: N x K, plain scales),
 * each dequantized as above, products summed in double, rounded once. */
int nvfp4ref_gemm(const uint8_t* qa, const uint8_t* sa, float alpha_a, const uint8_t* qb,
                  const uint8_t* sb, float alpha_b, int64_t M, int64_t N, int64_t K, float* d);

/* Error histogram of a rowwise copy over v = 6|x|/b (see the definition). */
int nvfp4ref_error_histogram(const uint16_t* x, int64_t M, int64_t N, int64_t ld, const uint8_t* q,
                             const uint8_t* s, float alpha, int nbins, uint64_t* hist);

#ifdef __cplusplus
}
#endif
#endif
