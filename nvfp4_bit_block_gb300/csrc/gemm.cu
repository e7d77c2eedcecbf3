// gemm.cu -- launch of the NVFP4 block-scaled GEMM (the kernel is in
// gemm_kernel.cuh): 128 x 256 output tiles when N is a multiple of 256, else
// 128 x 128.
#include "gemm_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  return (a.N % 256 == 0) ? gemmk::launch<256>(a, s) : gemmk::launch<128>(a, s);
}

}  // namespace nvfp4
