// quant1d_46mse.cu -- 4/6 quantize kernels with the mse selection rule.
#include "quant1d_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quant1d_46_mse(const QuantArgs& a, bool row, bool col, bool sr, cudaStream_t s) {
  return q1d::launch_family<true, kSelMSE>(a, row, col, sr, s);
}

}  // namespace nvfp4
