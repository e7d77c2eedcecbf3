/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 training quantizer.
 *
 * NVFP4 stores a tensor as 4-bit E2M1 codes, one FP8 E4M3 scale per block of
 * 16 elements and one FP32 tensor scale alpha.  The library turns a bf16
 * tensor X (M x N, row-major, leading dimension ld elements) into
 *   - a rowwise copy R: blocks of 16 consecutive elements of a row, and/or
 *   - a columnwise copy C: blocks of 16 consecutive elements of a column,
 *     stored as the transpose X^T (N x M, row-major),
 * both from one read of X.  Options: 16x16 2D block scales (weights), a
 * seeded 16-point random Hadamard transform (RHT), stochastic rounding (SR)
 * and the "4/6" adaptive block scale.
 *
 * Method sources (cited below by these tags):
 *   [P1] "Pretraining Large Language Models with NVFP4" (gist.science summary
 *        of arXiv 2509.25149): section 1 (16-element blocks with E4M3
 *        scales), section 2b (random Hadamard transforms, backward pass only),
 *        section 2c (2D block scaling), section 2d (stochastic rounding).
 *   [P2] "Four Over Six (4/6)" technical summary (gist.science, arXiv
 *        2512.02010): "Problem statement" (E2M1 steps 0.5/1/2, blocks scaled
 *        to [-6, 6]), "Methodology" (quantize each block at maximum 6 and at
 *        maximum 4, keep the one with the lower error; MAE, MSE or max-error
 *        rule), "Implementation details" (tensor scale over 256 instead of 448).
 *   [SK11] Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
 *        SC'11 (Philox4x32-10).
 *
 * Conventions for every call:
 *   - Pointers named *_dev are device pointers; the caller allocates and owns
 *     every buffer.  The library allocates nothing and keeps no state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream; a return of
 *     NVFP4_OK means the work was enqueued.
 *   - Argument errors are detected on the host and returned at once, before
 *     anything is enqueued.  Conditions that depend on device data (a non-finite
 *     or out-of-range amax) are written to the optional device status word.
 *   - Output layouts (all dense, row-major, no padding):
 *       q_row  M x N/2 bytes    codes of R; byte (r, j) holds element (r, 2j)
 *                               in its low nibble and (r, 2j+1) in its high
 *       s_row  M x N/16 bytes   E4M3 scale of block (r, c/16)
 *       q_col  N x M/2 bytes    codes of C = X^T; byte (c, j) holds elements
 *                               (2j, c) low and (2j+1, c) high
 *       s_col  N x M/16 bytes   E4M3 scale of block (c, r/16)
 *     A code is sign<<3 | index, index into the E2M1 magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6} ([P2] Problem statement).
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = -1,      /* a required pointer is NULL                            */
  NVFP4_ERR_SHAPE = -2,     /* N % 16 != 0; M % 16 != 0 with COLWISE or 2D; ld < N;
                               negative sizes; M or N above 2^31 - 1                  */
  NVFP4_ERR_ALIGN = -3,     /* x not 16-byte aligned or ld % 8 != 0; an output not
                               aligned to its access width                             */
  NVFP4_ERR_FLAGS = -4,     /* unknown bits; no copy requested; 2D with an RHT flag;
                               an RHT flag for a copy not requested; bad selector    */
  NVFP4_ERR_CUDA = -5,      /* a CUDA launch or copy failed                           */
  NVFP4_ERR_NONFINITE = -6, /* device status: amax is Inf or NaN                      */
  NVFP4_ERR_RANGE = -7,     /* device status: 0 < amax < 2^-100 (the per-block
                               reciprocal could overflow FP32)                        */
  NVFP4_ERR_PIPELINE = -8   /* device status: a tile copy into shared memory did not
                               complete within about a second; the kernel stopped
                               and the outputs are incomplete                         */
} nvfp4_status;

enum {
  NVFP4_ROWWISE = 1,  /* produce the rowwise copy R (1x16 blocks along rows)             */
  NVFP4_COLWISE = 2,  /* produce the columnwise copy C = X^T (1x16 blocks along columns) */
  NVFP4_2D = 4,       /* [P1] 2c: one scale per 16x16 tile shared by R and C             */
  NVFP4_RHT_ROW = 8,  /* [P1] 2b: 16-point RHT along rows before quantizing R            */
  NVFP4_RHT_COL = 16, /* [P1] 2b: 16-point RHT along columns before quantizing C         */
  NVFP4_SR = 32,      /* [P1] 2d: stochastic rounding (Philox4x32-10) instead of RN      */
  NVFP4_46 = 64,      /* [P2] Methodology: 4/6 adaptive block scale; alpha over 6*256    */
  NVFP4_SF_SWIZZLED = 128 /* scales in the tiled layout of block-scaled MMA operands (below) */
};

typedef enum {
  NVFP4_SEL_MAE = 0,   /* keep max-4 iff its sum of |error| is lower   ([P2] Methodology) */
  NVFP4_SEL_MSE = 1,   /* keep max-4 iff its sum of error^2 is lower                      */
  NVFP4_SEL_MAXERR = 2 /* keep max-4 iff its largest |error| is lower                     */
} nvfp4_select;

/*
 * nvfp4_amax -- tensor amax for each copy ([P2] Implementation details: the
 * global tensor scale comes from the tensor's largest magnitude).
 *
 *   x_dev     bf16 M x N, row stride ld elements; 16-byte aligned, ld % 8 == 0
 *   flags     the same flags the matching nvfp4_quantize call will get; only
 *             RHT_ROW / RHT_COL change the result
 *   rht_seed  seed of the RHT sign vector (used with RHT flags)
 *   amax_dev  float[2] (device): [0] = max |value| over what the R copy
 *             quantizes, [1] = the same for the C copy.  Without an RHT flag
 *             both are max|x|; with one, that copy's entry is the largest
 *             magnitude of its Hadamard-transformed 16-vectors.  A NaN input
 *             gives NaN, an Inf input Inf.  Overwritten, not accumulated.
 * Returns NVFP4_OK or a host-side error (nothing enqueued then).
 */
NVFP4_API int nvfp4_amax(const void* x_dev, int64_t M, int64_t N, int64_t ld, uint32_t flags,
               uint64_t rht_seed, float* amax_dev, void* stream);

/*
 * nvfp4_quantize -- one read of X, rowwise and/or columnwise NVFP4 outputs.
 *
 * Per copy k (0 = R, 1 = C): alpha_k = amax_k / 2688 (6*448), or
 * amax_k / 1536 (6*256) with NVFP4_46 ([P2] Implementation details).  Per
 * block of 16 values z (or 256 with 2D) and block maximum Q = 6:
 *   b = max|z|;  e = E4M3(b / (Q*alpha));  d = e*alpha;
 *   v = z * (1/d);  code = sign | round(min(|v|, Q))
 * with round = nearest (ties to even code) or, with NVFP4_SR, up with
 * probability (m-lo)/(hi-lo) ([P1] 2d).  With NVFP4_46 the block is also
 * quantized at Q = 4 and the candidate with the strictly lower error score is
 * kept ([P2] Methodology); the scale byte then tells which.
 *
 *   x_dev           bf16 M x N as for nvfp4_amax (must not change in between)
 *   amax_dev        float[2] written by nvfp4_amax on the same stream
 *   flags           NVFP4_* bits; at least one of ROWWISE / COLWISE
 *   sel             nvfp4_select, used with NVFP4_46
 *   sr_seed         Philox key for SR; the counter of element (r, c) is
 *                   counter_offset + r*N + c; R uses word 0, C word 1 (2D: both
 *                   word 0)
 *   rht_seed        Philox key of the RHT signs (counter (0,0,0,1), word 0)
 *   counter_offset  added to every SR counter (lets a row shard reproduce the
 *                   unsharded bits: offset = first_row * N)
 *   q_row, s_row    R outputs (required with ROWWISE, else ignored; may be NULL)
 *   q_col, s_col    C outputs (required with COLWISE, else ignored; may be NULL)
 *                   q_row/q_col 16-byte aligned, s_row/s_col 4-byte aligned
 *   alpha_dev       float[2] (device): alpha of R and C, always written
 *   status_dev      int (device) or NULL: set to NVFP4_ERR_NONFINITE or
 *                   NVFP4_ERR_RANGE when a requested copy's amax is not usable,
 *                   in which case no code or scale byte is written, or to
 *                   NVFP4_ERR_PIPELINE when a tile load timed out; left
 *                   untouched on success (the caller zeroes it)
 * With 2D, the tile scale is repeated in the 1x16 scale layouts (16 times in
 * s_row, 16 times in s_col) and C's codes are exactly the transpose of R's.
 *
 * Scale layouts.  Plain (default): s_row is M x N/16 row-major, s_col is
 * N x M/16 row-major.  With NVFP4_SF_SWIZZLED each copy's scale matrix
 * (R rows x C = K/16 scale columns: R = M, K = N for s_row; R = N, K = M for
 * s_col) is stored in tiles of 128 rows x 4 scale columns, 512 bytes each,
 * tiles in row-major order over the padded matrix (R rounded up to 128 rows,
 * C to 4 columns), and inside a tile scale (r, c) at byte
 * (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4 -- the order in which a
 * block-scaled tensor-core MMA (FP4 operand with one E4M3 scale per 16 values
 * along K) takes its scale factors, so a GEMM can read the scales directly.
 * The buffer then holds ceil(R/128)*128 * ceil(C/4)*4 bytes; entries of the
 * padding are not written (zero them if the consumer reads them).  Codes are
 * unaffected.  nvfp4_dequantize reads the plain layout only.
 */
NVFP4_API int nvfp4_quantize(const void* x_dev, int64_t M, int64_t N, int64_t ld, const float* amax_dev,
                   uint32_t flags, int sel, uint64_t sr_seed, uint64_t rht_seed,
                   uint64_t counter_offset, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                   uint8_t* s_col, float* alpha_dev, int* status_dev, void* stream);

/*
 * nvfp4_dequantize -- x^ = val(code) * (float(e) * alpha), the reconstruction
 * the 4/6 error of [P2] Methodology is measured against.
 *
 *   q_dev      rows x cols/2 code bytes (a q_row or q_col buffer)
 *   s_dev      rows x cols/16 scale bytes (the matching s_row or s_col)
 *   alpha_dev  one float (device): that copy's alpha (alpha_dev + 0 or + 1)
 *   out_dev    rows x cols, fp32 (out_is_bf16 = 0) or bf16 rounded to nearest
 *              even (out_is_bf16 = 1); 16-byte aligned
 * cols % 16 == 0.  With an RHT copy the result is in the transformed basis.
 */
NVFP4_API int nvfp4_dequantize(const uint8_t* q_dev, const uint8_t* s_dev, const float* alpha_dev,
                     int64_t rows, int64_t cols, int out_is_bf16, void* out_dev, void* stream);

/*
 * nvfp4_error_histogram -- where the rounding error of a rowwise copy sits
 * within its blocks (the 4/6 page's Problem statement: values between 4 and 6
 * at block scale 6, around scaled value 5, carry the damaging error).
 *
 *   x_dev      bf16 M x N (row stride ld elements), the tensor that was quantized
 *   q_dev      its rowwise codes (M x N/2), s_dev its rowwise scales in the
 *              plain layout (M x N/16), alpha_dev the copy's alpha (one float)
 *   nbins      1..1024 equal bins over v = 6|x|/b in [0, 6], b = the
 *              element's block maximum (bin = min(floor(v*nbins/6), nbins-1))
 *   hist_dev   unsigned 64-bit [3][nbins] on the device, ADDED to (zero it
 *              first): element counts; sums of e = 6|x - x^|/b in units of
 *              2^-24; sums of e*e in units of 2^-32 (each term truncated);
 *              x^ as nvfp4_dequantize reconstructs it.  Blocks with b = 0
 *              are skipped.  Integer sums: the result is exact and
 *              independent of the launch configuration.
 * Asynchronous on `stream`.  Errors: SHAPE (N % 16, ld < N, nbins out of
 * range), NULL, ALIGN (x 16-byte, q 8-byte, ld % 8), CUDA.
 */
NVFP4_API int nvfp4_error_histogram(const void* x_dev, int64_t M, int64_t N, int64_t ld, const uint8_t* q_dev,
                                    const uint8_t* s_dev, const float* alpha_dev, int nbins,
                                    unsigned long long* hist_dev, void* stream);

/*
 * nvfp4_gemm -- D = alpha_a * alpha_b * (A * B^T) on the FP4 tensor cores
 * ("NVFP4 revolutionizes AI training" headline page: Blackwell computes
 * matrix products on FP4 operands natively).
 *
 * A (M x K) and B (N x K) are NVFP4 operands as nvfp4_quantize writes them
 * with NVFP4_SF_SWIZZLED: packed codes with K contiguous (a rowwise copy, or
 * the columnwise copy of a tensor whose transpose is the operand) and E4M3
 * scales per 16 values along K in the tiled 128 x 4 layout.  Each product is
 * formed from val(code) * e4m3(scale) per operand, the sum over K is
 * accumulated in fp32 by the tensor cores, and the result is multiplied by
 * alpha_a * alpha_b (rounded once to fp32, then to bf16 with out_is_bf16)
 * -- the dequantized operands' product up to the order and rounding of the
 * fp32 accumulation.
 *
 *   qa_dev       M x K/2 code bytes (16-byte aligned)
 *   sfa_dev      tiled scales of A: M/128 * K/64 blocks of 512 bytes
 *                (16-byte aligned)
 *   alpha_a_dev  one float (device): A's tensor scale (the alpha of its copy)
 *   qb_dev, sfb_dev, alpha_b_dev   the same for B (N rows)
 *   out_is_bf16  0: D is fp32; 1: D is bf16 (round to nearest even)
 *   d_dev        M x N, row stride ldd elements (16-byte aligned, ldd >= N,
 *                ldd % 4 == 0 for fp32, ldd % 8 == 0 for bf16)
 *   status_dev   int (device) or NULL: set to NVFP4_ERR_PIPELINE if a tile
 *                copy or the tensor-core work did not complete within about
 *                a second (D is then incomplete); untouched on success
 * Shapes: M % 128 == 0, N % 128 == 0, K % 256 == 0, K > 0 (M or N = 0: no-op).
 * Asynchronous on `stream`.  Errors: SHAPE, NULL, ALIGN, CUDA.
 */
NVFP4_API int nvfp4_gemm(const uint8_t* qa_dev, const uint8_t* sfa_dev, const float* alpha_a_dev,
                         const uint8_t* qb_dev, const uint8_t* sfb_dev, const float* alpha_b_dev, int64_t M,
                         int64_t N, int64_t K, int out_is_bf16, void* d_dev, int64_t ldd, int* status_dev,
                         void* stream);

/* Human-readable name of a status value (static string). */
NVFP4_API const char* nvfp4_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
