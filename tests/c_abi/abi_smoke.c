/* Pure-C use of the library's C ABI (no Python, no PyTorch): one fused run
 * of the row-parallel layer on an exact-integer case, checked on the host.
 *
 * A and W hold values in {-1, 0, 1}, so every rank's partial over K/8 = 16
 * terms is an integer of magnitude <= 16 and the sum of the 8 partials is an
 * integer of magnitude <= 128: exact in bf16 and fp32 at every step, so the
 * output must equal the integer product A W computed here.  Exit status 0 on
 * success.  Build: cc abi_smoke.c -I<include> -L<lib> -lgemm_rs -lcudart.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gemm_rs.h"

enum { M = 64, N = 256, K = 128, R = GEMM_RS_WORLD, KR = K / GEMM_RS_WORLD };

static uint16_t bf16_of_int(int v) { /* small integers are exact in bf16 */
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}
static float float_of_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int main(void) {
  static int a[M][K], w[K][N];
  static uint16_t A[R][M][KR], W[R][KR][N], out[M][N];
  uint32_t seed = 12345u;
  for (int i = 0; i < M; ++i)
    for (int k = 0; k < K; ++k) {
      seed = seed * 1664525u + 1013904223u;
      a[i][k] = (int)((seed >> 16) % 3u) - 1;
    }
  for (int k = 0; k < K; ++k)
    for (int j = 0; j < N; ++j) {
      seed = seed * 1664525u + 1013904223u;
      w[k][j] = (int)((seed >> 16) % 3u) - 1;
    }
  for (int r = 0; r < R; ++r)
    for (int i = 0; i < M; ++i)
      for (int k = 0; k < KR; ++k) A[r][i][k] = bf16_of_int(a[i][r * KR + k]);
  for (int r = 0; r < R; ++r)
    for (int k = 0; k < KR; ++k)
      for (int j = 0; j < N; ++j) W[r][k][j] = bf16_of_int(w[r * KR + k][j]);

  gemm_rs_desc d;
  memset(&d, 0, sizeof(d));
  d.world = GEMM_RS_WORLD;
  d.M = M;
  d.N = N;
  d.K = K;
  gemm_rs_t plan = NULL;
  size_t ws_bytes = 0;
  int rc = gemm_rs_create(&d, &plan, &ws_bytes);
  if (rc != GEMM_RS_OK) {
    fprintf(stderr, "create: %s\n", gemm_rs_strerror(rc));
    return 1;
  }
  void *dA = NULL, *dW = NULL, *dOut = NULL, *ws = NULL;
  if (cudaMalloc(&dA, sizeof(A)) || cudaMalloc(&dW, sizeof(W)) || cudaMalloc(&dOut, sizeof(out)) ||
      cudaMalloc(&ws, ws_bytes)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 1;
  }
  cudaStream_t st;
  cudaStreamCreate(&st);
  rc = gemm_rs_run_host(plan, GEMM_RS_FUSED, A, W, out, dA, dW, dOut, ws, st);
  if (rc == GEMM_RS_OK) rc = gemm_rs_status(plan, st);
  if (rc != GEMM_RS_OK) {
    fprintf(stderr, "run: %s\n", gemm_rs_strerror(rc));
    return 1;
  }
  int bad = 0;
  for (int i = 0; i < M; ++i)
    for (int j = 0; j < N; ++j) {
      int s = 0;
      for (int k = 0; k < K; ++k) s += a[i][k] * w[k][j];
      if (float_of_bf16(out[i][j]) != (float)s && bad++ < 5)
        fprintf(stderr, "out[%d][%d] = %g, expected %d\n", i, j, float_of_bf16(out[i][j]), s);
    }
  gemm_rs_destroy(plan);
  cudaFree(dA);
  cudaFree(dW);
  cudaFree(dOut);
  cudaFree(ws);
  cudaStreamDestroy(st);
  if (bad) {
    fprintf(stderr, "%d mismatches\n", bad);
    return 1;
  }
  printf("c abi ok: %dx%dx%d exact\n", M, N, K);
  return 0;
}
