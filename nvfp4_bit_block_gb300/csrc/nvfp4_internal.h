// nvfp4_internal.h -- kernel launch interface shared by the library's own
// translation units (not part of the public C ABI).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

struct QuantArgs {
  const uint16_t* x;
  int64_t M, N, ld;
  const float* amax;  // [2]
  float* alpha;       // [2]
  int* status;        // nullable
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  uint64_t ctr_off;
  uint32_t sr_k0, sr_k1;
  uint32_t rht_k0, rht_k1;
  int sel;
  int rht_row, rht_col;
  int sf_swz;  // scales in the tiled block-scaled-MMA layout
};

struct AmaxArgs {
  const uint16_t* x;
  int64_t M, N, ld;
  uint32_t rht_k0, rht_k1;
  float* amax;  // [2], zeroed before the launch
};

struct DequantArgs {
  const uint8_t* q;
  const uint8_t* s;
  const float* alpha;
  int64_t rows, cols;
  int out_bf16;
  void* out;
};

struct HistArgs {
  const uint16_t* x;
  int64_t M, N, ld;
  const uint8_t* q;      // rowwise codes, M x N/2
  const uint8_t* s;      // rowwise scales, M x N/16 (plain layout)
  const float* alpha;    // the copy's alpha
  int nbins;
  unsigned long long* hist;  // [3][nbins], accumulated into
};

struct GemmArgs {
  const uint8_t* qa;    // M x K/2 codes (K contiguous)
  const uint8_t* sfa;   // tiled scales of A (128 x 4 tiles of 512 bytes)
  const float* alpha_a; // [1]
  const uint8_t* qb;    // N x K/2 codes
  const uint8_t* sfb;   // tiled scales of B
  const float* alpha_b; // [1]
  void* d;              // M x N, row stride ldd elements
  int64_t M, N, K, ldd;
  int out_bf16;         // D in bf16 (else fp32)
  int* status;          // nullable
};

// TMA boxes of the bf16 input: 64 columns (128 bytes, the swizzle span) x 64 rows.
constexpr int kBoxCols = 64;
constexpr int kBoxRows = 64;
cudaError_t make_tile_map(CUtensorMap* map, const uint16_t* x, int64_t M, int64_t N, int64_t ld);
// Packed FP4 codes (rows x row_bytes bytes, dense) read in 128-byte-swizzled
// boxes of box_bytes x box_rows.
cudaError_t make_codes_map(CUtensorMap* map, const uint8_t* q, int64_t rows, int64_t row_bytes, int box_bytes,
                           int box_rows);

// Grid of a persistent kernel on the current device: resident CTAs per SM
// (at `threads` threads and `smem` bytes of dynamic shared memory, which the
// kernel is first opted in to) times the SM count.  Computed once per device
// and kept in `cache` (one 64-slot array per kernel instantiation; atomic, so
// concurrent host threads may launch).
template <typename Kernel>
cudaError_t resident_grid(Kernel kern, int threads, int smem, std::atomic<int>* cache, int& cap) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < 64;
  cap = slot ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (cap > 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cap = (per_sm > 0 ? per_sm : 1) * sms;
  if (slot) cache[dev].store(cap, std::memory_order_relaxed);
  return cudaSuccess;
}

cudaError_t launch_amax(const AmaxArgs& a, bool rht_row, bool rht_col, cudaStream_t s);
cudaError_t launch_quant1d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t s);
// rowwise + columnwise, stochastic rounding, no 4/6, Hadamard on the columnwise copy or none
cudaError_t launch_quant1d_sr_rc(const QuantArgs& a, bool rht_col, cudaStream_t s);
cudaError_t launch_quant1d_46_mae(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s);
cudaError_t launch_quant1d_46_mse(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s);
cudaError_t launch_quant1d_46_max(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s);
cudaError_t launch_quant2d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_error_hist(const HistArgs& a, cudaStream_t s);
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);

}  // namespace nvfp4
