/* A plain C caller of the library: no Python, no PyTorch.  Device memory comes from the CUDA
 * runtime; every call goes through include/fge.h.
 *
 * Closed form checked: x = 1 everywhere (bf16), W = 1 everywhere (e4m3 code 0x38), weight
 * scale 1.  The per-tensor activation scale is amax / 448 = 1/448, so every activation code
 * is 448 and y[m, n] = sum_k 448 * 1 * (1/448) = K exactly, at a decode size (M = 16, the
 * swapped tile with the K split) and at a 128-row size (M = 300).  Also checked: a NULL
 * pointer is refused before anything runs, and the status strings are there.
 * Exit status 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "fge.h"

static int fail(const char* what) {
  fprintf(stderr, "c_abi: %s\n", what);
  return 1;
}

static int run_case(int64_t M, int64_t K, int64_t N, cudaStream_t s) {
  const uint16_t one_bf16 = 0x3F80u;
  const uint8_t one_e4m3 = 0x38u;
  uint16_t* hx = (uint16_t*)malloc((size_t)(M * K) * 2);
  uint8_t* hw = (uint8_t*)malloc((size_t)(N * K));
  uint16_t* hy = (uint16_t*)malloc((size_t)(M * N) * 2);
  if (!hx || !hw || !hy) return fail("host allocation");
  for (int64_t i = 0; i < M * K; ++i) hx[i] = one_bf16;
  memset(hw, one_e4m3, (size_t)(N * K));
  const float w_scale = 1.0f;

  void *dx, *dw, *dy, *dws, *dsw;
  const size_t ws_bytes = fge_workspace_bytes(FGE_OP_LINEAR_W8A8, M, K, N, 0, 0);
  if (cudaMalloc(&dx, (size_t)(M * K) * 2) != cudaSuccess ||
      cudaMalloc(&dw, (size_t)(N * K)) != cudaSuccess ||
      cudaMalloc(&dy, (size_t)(M * N) * 2) != cudaSuccess ||
      cudaMalloc(&dws, ws_bytes) != cudaSuccess || cudaMalloc(&dsw, sizeof(float)) != cudaSuccess)
    return fail("cudaMalloc");
  cudaMemcpy(dx, hx, (size_t)(M * K) * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dw, hw, (size_t)(N * K), cudaMemcpyHostToDevice);
  cudaMemcpy(dsw, &w_scale, sizeof(float), cudaMemcpyHostToDevice);
  cudaMemset(dy, 0, (size_t)(M * N) * 2);

  if (fge_linear_w8a8(NULL, M, K, (const uint8_t*)dw, (const float*)dsw, N, dy, dws, ws_bytes,
                      (fge_stream_t)s) != FGE_ERR_INVALID_ARG)
    return fail("a NULL activation pointer was not refused");
  fge_status st = fge_linear_w8a8(dx, M, K, (const uint8_t*)dw, (const float*)dsw, N, dy, dws,
                                  ws_bytes, (fge_stream_t)s);
  if (st != FGE_OK) {
    fprintf(stderr, "c_abi: fge_linear_w8a8: %s\n", fge_status_string(st));
    return 1;
  }
  int32_t dev_status = -1;
  if (fge_read_device_status(dws, (fge_stream_t)s, &dev_status) != FGE_OK || dev_status != 0)
    return fail("device status");
  cudaMemcpy(hy, dy, (size_t)(M * N) * 2, cudaMemcpyDeviceToHost);
  /* K = 256 or 2560 as bf16: exact (both are 8-bit-mantissa values times a power of two) */
  float want = (float)K;
  uint32_t wb;
  memcpy(&wb, &want, 4);
  const uint16_t want_bf16 = (uint16_t)(wb >> 16);
  for (int64_t i = 0; i < M * N; ++i) {
    if (hy[i] != want_bf16) {
      fprintf(stderr, "c_abi: M=%lld y[%lld] = 0x%04x, want 0x%04x\n", (long long)M,
              (long long)i, hy[i], want_bf16);
      return 1;
    }
  }
  cudaFree(dx);
  cudaFree(dw);
  cudaFree(dy);
  cudaFree(dws);
  cudaFree(dsw);
  free(hx);
  free(hw);
  free(hy);
  return 0;
}

int main(void) {
  if (fge_init(0) != FGE_OK) return fail("fge_init");
  if (fge_status_string(FGE_OK) == NULL || fge_status_string(FGE_ERR_INVALID_ARG) == NULL)
    return fail("status strings");
  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) return fail("stream");
  if (run_case(16, 2560, 6656, s)) return 1;
  if (run_case(300, 256, 384, s)) return 1;
  cudaStreamDestroy(s);
  printf("c_abi ok: fge_linear_w8a8 closed form at M = 16 and M = 300\n");
  return 0;
}
