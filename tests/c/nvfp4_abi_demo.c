/* nvfp4_abi_demo.c -- the C ABI used from plain C (no Python, no torch).
 *
 * Without a GPU: checks that argument errors come back as documented.
 * With a GPU: quantizes a 64 x 64 bf16 tensor whose every value is 1.5 and
 * checks the result worked out by hand from the NVFP4 recipe:
 *   standard (alpha = amax / 2688): t = 1.5 / (6 alpha) = 448 -> scale byte
 *   0x7E, d = 448 alpha = 0.25, every value scales to 6.0 -> code 7;
 *   4/6 (alpha = amax / 1536): max-6 scale 256 (byte 0x78), values at 6.0,
 *   error 0; max-4 scale 384 (byte 0x7C), values at 4.0, error 0; the tie
 *   keeps max 6 -> codes 7, byte 0x78.
 * Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "nvfp4.h"

#define CHECK(cond, msg)                       \
  do {                                         \
    if (!(cond)) {                             \
      fprintf(stderr, "FAILED: %s\n", (msg));  \
      return 1;                                \
    }                                          \
  } while (0)

static int host_checks(void) {
  static uint16_t x[16];
  float amax[2];
  CHECK(strcmp(nvfp4_strerror(NVFP4_OK), "ok") == 0, "strerror(OK)");
  CHECK(nvfp4_amax(x, 1, 16, 16, 0, 0, amax, NULL) == NVFP4_ERR_FLAGS, "no copy requested");
  CHECK(nvfp4_amax(x, 1, 24, 24, NVFP4_ROWWISE, 0, amax, NULL) == NVFP4_ERR_SHAPE, "N % 16");
  CHECK(nvfp4_amax(x, 1, 16, 16, NVFP4_ROWWISE, 0, NULL, NULL) == NVFP4_ERR_NULL, "null amax");
  CHECK(nvfp4_quantize(x, 1, 16, 16, amax, NVFP4_ROWWISE | NVFP4_2D | NVFP4_RHT_ROW, 0, 0, 0, 0, NULL, NULL,
                       NULL, NULL, amax, NULL, NULL) == NVFP4_ERR_FLAGS,
        "2D with RHT");
  return 0;
}

static int gpu_checks(void) {
  enum { M = 64, N = 64 };
  static uint16_t hx[M * N];
  static uint8_t hq[M * N / 2], hs[M * N / 16];
  for (int i = 0; i < M * N; ++i) hx[i] = 0x3FC0; /* bf16 1.5 */
  void* dx;
  float *damax, *dalpha;
  uint8_t *dq, *ds, *dqc, *dsc;
  int* dstatus;
  CHECK(cudaMalloc(&dx, sizeof hx) == cudaSuccess, "cudaMalloc");
  cudaMalloc((void**)&damax, 2 * sizeof(float));
  cudaMalloc((void**)&dalpha, 2 * sizeof(float));
  cudaMalloc((void**)&dq, sizeof hq);
  cudaMalloc((void**)&ds, sizeof hs);
  cudaMalloc((void**)&dqc, sizeof hq);
  cudaMalloc((void**)&dsc, sizeof hs);
  cudaMalloc((void**)&dstatus, sizeof(int));
  cudaMemcpy(dx, hx, sizeof hx, cudaMemcpyHostToDevice);
  for (int variant = 0; variant < 2; ++variant) {
    const uint32_t flags = NVFP4_ROWWISE | NVFP4_COLWISE | (variant ? NVFP4_46 : 0);
    cudaMemset(dstatus, 0, sizeof(int));
    CHECK(nvfp4_amax(dx, M, N, N, flags, 0, damax, NULL) == NVFP4_OK, "nvfp4_amax");
    CHECK(nvfp4_quantize(dx, M, N, N, damax, flags, NVFP4_SEL_MAE, 1, 2, 0, dq, ds, dqc, dsc, dalpha, dstatus,
                         NULL) == NVFP4_OK,
          "nvfp4_quantize");
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "synchronize");
    int status = -1;
    float amax[2];
    cudaMemcpy(&status, dstatus, sizeof(int), cudaMemcpyDeviceToHost);
    cudaMemcpy(amax, damax, sizeof amax, cudaMemcpyDeviceToHost);
    CHECK(status == 0 && amax[0] == 1.5f && amax[1] == 1.5f, "status and amax");
    const uint8_t want_scale = variant ? 0x78 : 0x7E;
    for (int copy = 0; copy < 2; ++copy) {
      cudaMemcpy(hq, copy ? dqc : dq, sizeof hq, cudaMemcpyDeviceToHost);
      cudaMemcpy(hs, copy ? dsc : ds, sizeof hs, cudaMemcpyDeviceToHost);
      for (int i = 0; i < M * N / 2; ++i) CHECK(hq[i] == 0x77, "codes are 6.0");
      for (int i = 0; i < M * N / 16; ++i) CHECK(hs[i] == want_scale, "scale bytes");
    }
  }
  printf("gpu checks passed\n");
  return 0;
}

int main(void) {
  if (host_checks()) return 1;
  printf("host checks passed\n");
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    printf("no GPU: skipped the device part\n");
    return 0;
  }
  return gpu_checks();
}
