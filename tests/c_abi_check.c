/* A plain C99 program using the library only through include/sk_gemm.h and the CUDA runtime:
 * it plans a Stream-K launch, runs sk_gemm_bf16 on device buffers and checks the result
 * (A = 1, B = 1, fp32 bias[n] = n  =>  fp32 C[m][n] = K + n, exact).
 * Without a GPU it checks only the host-side calls.  Exit status 0 means success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "sk_gemm.h"

#define M 300
#define N 264
#define K 512

static uint16_t bf16_of(float x) { /* exact for the small integers used here */
  union { float f; uint32_t u; } v;
  v.f = x;
  return (uint16_t)(v.u >> 16);
}

int main(void) {
  sk_plan_t plan;
  if (sk_plan(0, M, N, K, 0, SK_MODE_STREAMK, 152, NULL, &plan) != SK_OK || plan.tiles < 1) {
    fprintf(stderr, "sk_plan failed\n");
    return 1;
  }
  int devices = 0;
  if (cudaGetDeviceCount(&devices) != cudaSuccess || devices == 0) {
    /* no GPU: a valid call must be refused cleanly, not crash */
    sk_status_t st = sk_gemm_bf16((void*)0x100000, (void*)0x100000, NULL, (void*)0x100000,
                                  SK_BF16, M, N, K, 0, SK_MODE_STREAMK, NULL);
    printf("no GPU: sk_gemm_bf16 -> %s\n", sk_status_string(st));
    return st == SK_ERR_UNSUPPORTED ? 0 : 1;
  }
  uint16_t* hA = (uint16_t*)malloc(sizeof(uint16_t) * M * K);
  uint16_t* hB = (uint16_t*)malloc(sizeof(uint16_t) * K * N);
  float* hbias = (float*)malloc(sizeof(float) * N);
  float* hC = (float*)malloc(sizeof(float) * M * N);
  for (int i = 0; i < M * K; ++i) hA[i] = bf16_of(1.0f);
  for (int i = 0; i < K * N; ++i) hB[i] = bf16_of(1.0f);
  for (int n = 0; n < N; ++n) hbias[n] = (float)n;
  void *dA, *dB, *dbias, *dC;
  if (cudaMalloc(&dA, sizeof(uint16_t) * M * K) != cudaSuccess ||
      cudaMalloc(&dB, sizeof(uint16_t) * K * N) != cudaSuccess ||
      cudaMalloc(&dbias, sizeof(float) * N) != cudaSuccess ||
      cudaMalloc(&dC, sizeof(float) * M * N) != cudaSuccess)
    return 2;
  cudaMemcpy(dA, hA, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, hB, sizeof(uint16_t) * K * N, cudaMemcpyHostToDevice);
  cudaMemcpy(dbias, hbias, sizeof(float) * N, cudaMemcpyHostToDevice);
  const sk_mode_t modes[5] = {SK_MODE_DP, SK_MODE_PERSISTENT, SK_MODE_STREAMK, SK_MODE_HYBRID,
                              SK_MODE_AUTO};
  for (int i = 0; i < 5; ++i) {
    cudaMemset(dC, 0, sizeof(float) * M * N);
    sk_status_t st = sk_gemm_bf16(dA, dB, dbias, dC, SK_F32, M, N, K, 7, modes[i], NULL);
    if (st == SK_OK) st = sk_stream_status(NULL);
    if (st != SK_OK) {
      fprintf(stderr, "mode %d: %s\n", (int)modes[i], sk_status_string(st));
      return 3;
    }
    cudaMemcpy(hC, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
    for (int m = 0; m < M; ++m)
      for (int n = 0; n < N; ++n)
        if (hC[m * N + n] != (float)(K + n)) {
          fprintf(stderr, "mode %d: C[%d][%d] = %g, want %d\n", (int)modes[i], m, n,
                  (double)hC[m * N + n], K + n);
          return 4;
        }
  }
  printf("C ABI check passed (%d tiles, %d k-iterations per tile)\n", (int)plan.tiles,
         (int)plan.iters);
  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dbias);
  cudaFree(dC);
  free(hA);
  free(hB);
  free(hbias);
  free(hC);
  sk_workspace_release_all();
  return 0;
}
