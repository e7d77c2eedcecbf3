// tmap.cu -- host-side tensor maps for the TMA tile loads.
//
// The bf16 input X (M x N, row stride ld elements) is described as a 2D
// tensor {N, M} and read in 64 x 64 boxes (128 bytes per box row, the 128-byte
// swizzle span); elements outside the tensor arrive as zeros.  The encoder is
// fetched from the driver once through the runtime, so the library does not
// link the driver API.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>

#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 load_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t make_tile_map(CUtensorMap* map, const uint16_t* x, int64_t M, int64_t N, int64_t ld) {
  std::memset(map, 0, sizeof(*map));
  if (M <= 0 || N <= 0) return cudaSuccess;  // nothing is loaded
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = load_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
  const cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBoxRows};
  const cuuint32_t elem_strides[2] = {1u, 1u};
  const CUresult r =
      encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, elem_strides,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_codes_map(CUtensorMap* map, const uint8_t* q, int64_t rows, int64_t row_bytes, int box_bytes,
                           int box_rows) {
  std::memset(map, 0, sizeof(*map));
  if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = load_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  const cuuint32_t elem_strides[2] = {1u, 1u};
  const CUresult r =
      encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, elem_strides,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace nvfp4
