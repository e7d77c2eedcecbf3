// tma.cuh -- Tensor Memory Accelerator tile loads completed on an mbarrier.
//
// One elected thread arms a shared-memory mbarrier with the byte count of a
// tile (mbarrier.arrive.expect_tx) and issues the 2D bulk tensor copies
// (cp.async.bulk.tensor) that deliver the tile; every consumer thread waits on
// the barrier's phase parity.  Waits are bounded: after about a second the
// wait reports failure instead of spinning on, so a copy that never arrives
// turns into a status value the host can read and the context stays usable.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace nvfp4 {
namespace tma {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second of %globaltimer
constexpr uint32_t kWaitLimitPolls = 1u << 26;    // backstop on the number of polls

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (the TMA unit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// Box (x = innermost coordinate, y) of the tensor described by `map` into
// shared memory at `dst`; completion is counted in bytes on `bar`.
__device__ __forceinline__ void load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false after the limit.
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1; i < kWaitLimitPolls; ++i) {
    if (try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

}  // namespace tma
}  // namespace nvfp4
