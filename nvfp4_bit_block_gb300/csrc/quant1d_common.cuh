#pragma once
// quant1d_common.cuh -- what the 1x16-block quantize kernels share: the tile
// shape and CTA size, the per-copy scale constants and the prologue (alpha of
// each copy, the amax status, the shared-memory alignment check).
//
// Sources: "Four Over Six (4/6)" technical summary (Implementation details:
// alpha over 6 * 256 with 4/6) and "Pretraining Large Language Models with
// NVFP4" section 1 (the two-level scale: alpha and the E4M3 block scales).
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"
#include "tile_pipeline.cuh"
#include "tma.cuh"

namespace nvfp4 {
namespace q1d {

using tile::kTM;
using tile::kTN;
constexpr int kBlockThreads = 256;

// Per-copy scale constants: den = Q*alpha and its correctly rounded
// reciprocal for Q = 6 and Q = 4, and the shared (d, 1/d) table of alpha.
struct CopyScales {
  float den6, rden6, den4, rden4;
  const float2* tbl;
};

__device__ __forceinline__ CopyScales make_scales(float alpha, const float2* tbl) {
  CopyScales c;
  c.den6 = __fmul_rn(6.0f, alpha);
  c.den4 = __fmul_rn(4.0f, alpha);
  c.rden6 = (c.den6 != 0.0f) ? __frcp_rn(c.den6) : 0.0f;
  c.rden4 = (c.den4 != 0.0f) ? __frcp_rn(c.den4) : 0.0f;
  c.tbl = tbl;
  return c;
}

// a2 and the checks every 1D kernel makes first: alpha of each copy (block 0
// writes both), the status of each produced copy's amax, and the 1 KB
// alignment of the dynamic shared memory that the 128-byte swizzle needs.
// False when the kernel must stop; block 0 has recorded why.
__device__ __forceinline__ bool begin_tensor(const QuantArgs& a, bool row, bool col, float den, const uint8_t* smem,
                                             float& alpha_r, float& alpha_c) {
  const float A_r = a.amax[0], A_c = a.amax[1];
  alpha_r = __fdiv_rn(A_r, den);
  alpha_c = __fdiv_rn(A_c, den);
  const int st_r = row ? amax_status(A_r) : 0;
  const int st_c = col ? amax_status(A_c) : 0;
  const bool misaligned = (tile::smem_u32(smem) & 1023u) != 0u;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.alpha[0] = alpha_r;
    a.alpha[1] = alpha_c;
    if ((st_r || st_c) && a.status) *a.status = st_r ? st_r : st_c;
    if (misaligned && !(st_r || st_c) && a.status) *a.status = kStatusPipeline;
  }
  return !(st_r || st_c || misaligned);
}

}  // namespace q1d
}  // namespace nvfp4
