// quant1d_sr.cu -- launcher of the stochastic-rounding rowwise + columnwise
// 1D kernel (quant1d_sr_kernel.cuh), in its own translation unit so that it
// compiles in parallel with the other quantize kernels.
#include "quant1d_sr_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quant1d_sr_rc(const QuantArgs& a, bool rht_col, cudaStream_t s) {
  return rht_col ? q1d::launch_sr_rc<true>(a, s) : q1d::launch_sr_rc<false>(a, s);
}

}  // namespace nvfp4
