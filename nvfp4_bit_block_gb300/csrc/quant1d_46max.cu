// quant1d_46max.cu -- 4/6 quantize kernels with the max selection rule.
#include "quant1d_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quant1d_46_max(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s) {
  return q1d::launch_family<true, kSelMax>(a, row, col, sr, s);
}

}  // namespace nvfp4
