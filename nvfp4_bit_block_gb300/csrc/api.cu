// api.cu -- the C ABI declared in include/nvfp4.h: host-side argument
// validation, flag decoding and kernel dispatch.  Nothing here allocates
// memory or keeps state; every call enqueues work on the caller's stream.
#include "nvfp4.h"

#include <cuda_runtime.h>

#include <cstdint>

#include "nvfp4_internal.h"

namespace {

constexpr uint32_t kKnownFlags = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_2D | NVFP4_RHT_ROW | NVFP4_RHT_COL | NVFP4_SR |
                                  NVFP4_46 | NVFP4_SF_SWIZZLED;

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int check_flags(uint32_t flags) {
  if (flags & ~kKnownFlags) return NVFP4_ERR_FLAGS;
  if (!(flags & (NVFP4_ROWWISE | NVFP4_COLWISE))) return NVFP4_ERR_FLAGS;
  if ((flags & NVFP4_2D) && (flags & (NVFP4_RHT_ROW | NVFP4_RHT_COL))) return NVFP4_ERR_FLAGS;
  if ((flags & NVFP4_RHT_ROW) && !(flags & NVFP4_ROWWISE)) return NVFP4_ERR_FLAGS;
  if ((flags & NVFP4_RHT_COL) && !(flags & NVFP4_COLWISE)) return NVFP4_ERR_FLAGS;
  return NVFP4_OK;
}

int check_shape(int64_t M, int64_t N, int64_t ld, uint32_t flags) {
  if (M < 0 || N < 0) return NVFP4_ERR_SHAPE;
  if (N % 16) return NVFP4_ERR_SHAPE;
  if ((flags & (NVFP4_COLWISE | NVFP4_2D)) && (M % 16)) return NVFP4_ERR_SHAPE;
  if (ld < N) return NVFP4_ERR_SHAPE;
  if (ld % 8) return NVFP4_ERR_ALIGN;
  // tile coordinates of the TMA copies are 32-bit
  if (M > INT32_MAX || N > INT32_MAX) return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

}  // namespace

extern "C" {

int nvfp4_amax(const void* x_dev, int64_t M, int64_t N, int64_t ld, uint32_t flags,
               uint64_t rht_seed, float* amax_dev, void* stream) {
  int st = check_flags(flags);
  if (st) return st;
  st = check_shape(M, N, ld, flags);
  if (st) return st;
  if (!amax_dev || (!x_dev && M > 0 && N > 0)) return NVFP4_ERR_NULL;
  if (!aligned(amax_dev, 4) || (x_dev && !aligned(x_dev, 16))) return NVFP4_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(amax_dev, 0, 2 * sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (M == 0 || N == 0) return NVFP4_OK;
  nvfp4::AmaxArgs a;
  a.x = static_cast<const uint16_t*>(x_dev);
  a.M = M;
  a.N = N;
  a.ld = ld;
  a.rht_k0 = (uint32_t)rht_seed;
  a.rht_k1 = (uint32_t)(rht_seed >> 32);
  a.amax = amax_dev;
  return launch_status(
      nvfp4::launch_amax(a, (flags & NVFP4_RHT_ROW) != 0, (flags & NVFP4_RHT_COL) != 0, s));
}

int nvfp4_quantize(const void* x_dev, int64_t M, int64_t N, int64_t ld, const float* amax_dev,
                   uint32_t flags, int sel, uint64_t sr_seed, uint64_t rht_seed,
                   uint64_t counter_offset, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                   uint8_t* s_col, float* alpha_dev, int* status_dev, void* stream) {
  int st = check_flags(flags);
  if (st) return st;
  if ((flags & NVFP4_46) && (sel < NVFP4_SEL_MAE || sel > NVFP4_SEL_MAXERR)) return NVFP4_ERR_FLAGS;
  st = check_shape(M, N, ld, flags);
  if (st) return st;
  const bool row = (flags & NVFP4_ROWWISE) != 0, col = (flags & NVFP4_COLWISE) != 0;
  const bool nonempty = M > 0 && N > 0;
  if (!amax_dev || !alpha_dev) return NVFP4_ERR_NULL;
  if (nonempty) {
    if (!x_dev) return NVFP4_ERR_NULL;
    if (row && (!q_row || !s_row)) return NVFP4_ERR_NULL;
    if (col && (!q_col || !s_col)) return NVFP4_ERR_NULL;
  }
  if ((x_dev && !aligned(x_dev, 16)) || !aligned(amax_dev, 4) || !aligned(alpha_dev, 4) ||
      (status_dev && !aligned(status_dev, 4)))
    return NVFP4_ERR_ALIGN;
  if (row && ((q_row && !aligned(q_row, 16)) || (s_row && !aligned(s_row, 4)))) return NVFP4_ERR_ALIGN;
  if (col && ((q_col && !aligned(q_col, 16)) || (s_col && !aligned(s_col, 4)))) return NVFP4_ERR_ALIGN;

  nvfp4::QuantArgs a;
  a.x = static_cast<const uint16_t*>(x_dev);
  a.M = M;
  a.N = N;
  a.ld = ld;
  a.amax = amax_dev;
  a.alpha = alpha_dev;
  a.status = status_dev;
  a.q_row = row ? q_row : nullptr;
  a.s_row = row ? s_row : nullptr;
  a.q_col = col ? q_col : nullptr;
  a.s_col = col ? s_col : nullptr;
  a.ctr_off = counter_offset;
  a.sr_k0 = (uint32_t)sr_seed;
  a.sr_k1 = (uint32_t)(sr_seed >> 32);
  a.rht_k0 = (uint32_t)rht_seed;
  a.rht_k1 = (uint32_t)(rht_seed >> 32);
  a.sel = (flags & NVFP4_46) ? sel : NVFP4_SEL_MAE;
  a.rht_row = (flags & NVFP4_RHT_ROW) ? 1 : 0;
  a.rht_col = (flags & NVFP4_RHT_COL) ? 1 : 0;
  a.sf_swz = (flags & NVFP4_SF_SWIZZLED) ? 1 : 0;
  const bool q46 = (flags & NVFP4_46) != 0, sr = (flags & NVFP4_SR) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (flags & NVFP4_2D) return launch_status(nvfp4::launch_quant2d(a, row, col, q46, sr, s));
  return launch_status(nvfp4::launch_quant1d(a, row, col, q46, sr, s));
}

int nvfp4_dequantize(const uint8_t* q_dev, const uint8_t* s_dev, const float* alpha_dev,
                     int64_t rows, int64_t cols, int out_is_bf16, void* out_dev, void* stream) {
  if (rows < 0 || cols < 0 || cols % 16) return NVFP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!q_dev || !s_dev || !alpha_dev || !out_dev) return NVFP4_ERR_NULL;
  if (!aligned(q_dev, 8) || !aligned(alpha_dev, 4) || !aligned(out_dev, 16)) return NVFP4_ERR_ALIGN;
  nvfp4::DequantArgs a;
  a.q = q_dev;
  a.s = s_dev;
  a.alpha = alpha_dev;
  a.rows = rows;
  a.cols = cols;
  a.out_bf16 = out_is_bf16 ? 1 : 0;
  a.out = out_dev;
  return launch_status(nvfp4::launch_dequant(a, static_cast<cudaStream_t>(stream)));
}

int nvfp4_error_histogram(const void* x_dev, int64_t M, int64_t N, int64_t ld, const uint8_t* q_dev,
                          const uint8_t* s_dev, const float* alpha_dev, int nbins, unsigned long long* hist_dev,
                          void* stream) {
  if (M < 0 || N < 0 || N % 16 || ld < N) return NVFP4_ERR_SHAPE;
  if (nbins < 1 || nbins > 1024) return NVFP4_ERR_SHAPE;
  if (!hist_dev) return NVFP4_ERR_NULL;
  if (M == 0 || N == 0) return NVFP4_OK;
  if (!x_dev || !q_dev || !s_dev || !alpha_dev) return NVFP4_ERR_NULL;
  if (!aligned(x_dev, 16) || ld % 8 || !aligned(q_dev, 8) || !aligned(alpha_dev, 4) || !aligned(hist_dev, 8))
    return NVFP4_ERR_ALIGN;
  nvfp4::HistArgs a;
  a.x = static_cast<const uint16_t*>(x_dev);
  a.M = M;
  a.N = N;
  a.ld = ld;
  a.q = q_dev;
  a.s = s_dev;
  a.alpha = alpha_dev;
  a.nbins = nbins;
  a.hist = hist_dev;
  return launch_status(nvfp4::launch_error_hist(a, static_cast<cudaStream_t>(stream)));
}

int nvfp4_gemm(const uint8_t* qa_dev, const uint8_t* sfa_dev, const float* alpha_a_dev, const uint8_t* qb_dev,
               const uint8_t* sfb_dev, const float* alpha_b_dev, int64_t M, int64_t N, int64_t K, int out_is_bf16,
               void* d_dev, int64_t ldd, int* status_dev, void* stream) {
  if (M < 0 || N < 0 || K < 0 || M % 128 || N % 128 || K % 256 || ldd < N) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (M == 0 || N == 0) return NVFP4_OK;
  if (K == 0) return NVFP4_ERR_SHAPE;
  if (!qa_dev || !sfa_dev || !alpha_a_dev || !qb_dev || !sfb_dev || !alpha_b_dev || !d_dev) return NVFP4_ERR_NULL;
  if (!aligned(qa_dev, 16) || !aligned(qb_dev, 16) || !aligned(sfa_dev, 16) || !aligned(sfb_dev, 16) ||
      !aligned(d_dev, 16) || ldd % (out_is_bf16 ? 8 : 4) || !aligned(alpha_a_dev, 4) || !aligned(alpha_b_dev, 4) ||
      (status_dev && !aligned(status_dev, 4)))
    return NVFP4_ERR_ALIGN;
  nvfp4::GemmArgs a;
  a.qa = qa_dev;
  a.sfa = sfa_dev;
  a.alpha_a = alpha_a_dev;
  a.qb = qb_dev;
  a.sfb = sfb_dev;
  a.alpha_b = alpha_b_dev;
  a.d = d_dev;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldd = ldd;
  a.out_bf16 = out_is_bf16 ? 1 : 0;
  a.status = status_dev;
  return launch_status(nvfp4::launch_gemm(a, static_cast<cudaStream_t>(stream)));
}

const char* nvfp4_strerror(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_NULL: return "a required pointer is NULL";
    case NVFP4_ERR_SHAPE: return "bad shape (N % 16, M % 16 with COLWISE/2D, ld < N, or M, N beyond 2^31 - 1)";
    case NVFP4_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case NVFP4_ERR_FLAGS: return "invalid flag combination or selection rule";
    case NVFP4_ERR_CUDA: return "CUDA launch failed";
    case NVFP4_ERR_NONFINITE: return "amax is Inf or NaN";
    case NVFP4_ERR_RANGE: return "amax below 2^-100";
    case NVFP4_ERR_PIPELINE: return "a tile copy did not arrive within the wait limit";
    default: return "unknown status";
  }
}

}  // extern "C"
