// quant1d.cu -- dispatch of the 1x16-block quantize kernels (the kernel
// itself is in quant1d_kernel.cuh).  The 4/6 variants are instantiated per
// selection rule in their own translation units so that each kernel holds
// exactly one rule's code and the units compile in parallel.
#include "quant1d_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quant1d(const QuantArgs& a, bool row, bool col, bool q46, bool sr, cudaStream_t s) {
  if (!q46) return q1d::launch_family<false, kSelMAE>(a, row, col, sr, s);
  if (a.sel == kSelMSE) return launch_quant1d_46_mse(a, row, col, sr, s);
  if (a.sel == kSelMax) return launch_quant1d_46_max(a, row, col, sr, s);
  return launch_quant1d_46_mae(a, row, col, sr, s);
}

}  // namespace nvfp4
