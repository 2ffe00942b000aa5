/*
 * c_abi_example.c -- drives libmxg.so through include/mxg.h from plain C:
 * device buffers from cudaMalloc, group offsets -> MXFP8 grouped quantize
 * (activations, both copies; weights, rowwise) -> grouped GEMM fprop, all on
 * one stream, then checks the result of a case with an exact answer.
 *
 * Case: G = 2 experts, K = N = 128, group rows {128, 128}.  Activation row m
 * is one-hot at column m % 128 (value 1), expert g's weight W_g[n, k] =
 * (n + 3k + 5g) % 9 - 4 (small integers, exactly representable), so the
 * output is exact: C[m, n] = W_g[n, m % 128] with g = m / 128.
 * Exit status 0 on success.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mxg.h"

static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16); /* the test values are exact in bf16 */
}

#define CK(x)                                                              \
  do {                                                                     \
    cudaError_t e_ = (x);                                                  \
    if (e_ != cudaSuccess) {                                               \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));             \
      return 2;                                                            \
    }                                                                      \
  } while (0)
#define MK(x)                                                              \
  do {                                                                     \
    mxg_status_t s_ = (x);                                                 \
    if (s_ != MXG_OK) {                                                    \
      fprintf(stderr, "%s: %s\n", #x, mxg_status_string(s_));              \
      return 3;                                                            \
    }                                                                      \
  } while (0)

int main(void) {
  const int G = 2, K = 128, N = 128, M = 256;
  uint16_t* hx = calloc((size_t)M * K, 2);
  uint16_t* hw = malloc((size_t)G * N * K * 2);
  float* hc = malloc((size_t)M * N * 4);
  int32_t hsizes[2] = {128, 128}, hst = 0;
  for (int m = 0; m < M; ++m) hx[(size_t)m * K + (m % 128)] = f32_to_bf16(1.0f);
  for (int g = 0; g < G; ++g)
    for (int n = 0; n < N; ++n)
      for (int k = 0; k < K; ++k)
        hw[((size_t)g * N + n) * K + k] = f32_to_bf16((float)((n + 3 * k + 5 * g) % 9 - 4));

  void *dx, *dw, *dsizes, *dws, *dst, *dqx, *dsfx, *dqxc, *dsfxc, *dqw, *dsfw, *dc;
  CK(cudaMalloc(&dx, (size_t)M * K * 2));
  CK(cudaMalloc(&dw, (size_t)G * N * K * 2));
  CK(cudaMalloc(&dsizes, sizeof(hsizes)));
  CK(cudaMalloc(&dws, mxg_offsets_workspace_bytes(G)));
  CK(cudaMalloc(&dst, 4));
  CK(cudaMalloc(&dqx, (size_t)M * K));
  CK(cudaMalloc(&dsfx, (size_t)M * K / 32));
  CK(cudaMalloc(&dqxc, (size_t)M * K));
  CK(cudaMalloc(&dsfxc, (size_t)M * K / 32));
  CK(cudaMalloc(&dqw, (size_t)G * N * K));
  CK(cudaMalloc(&dsfw, (size_t)G * N * K / 32));
  CK(cudaMalloc(&dc, (size_t)M * N * 4));
  cudaStream_t stream;
  CK(cudaStreamCreate(&stream));
  CK(cudaMemcpy(dx, hx, (size_t)M * K * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dw, hw, (size_t)G * N * K * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dsizes, hsizes, sizeof(hsizes), cudaMemcpyHostToDevice));
  CK(cudaMemset(dst, 0, 4));

  mxg_stream_t s = (mxg_stream_t)stream;
  MK(mxg_group_offsets(dsizes, 0, G, 1, K, M, (int64_t*)dws, (int32_t*)dst, s));
  MK(mxg_group_quantize(MXG_MXFP8_E4M3, MXG_BOTH, dx, M, K, (const int64_t*)dws, G, dqx,
                        (uint8_t*)dsfx, dqxc, (uint8_t*)dsfxc, NULL, NULL, (int32_t*)dst, s));
  MK(mxg_group_quantize(MXG_MXFP8_E4M3, MXG_ROWWISE, dw, (int64_t)G * N, K, NULL, G, dqw,
                        (uint8_t*)dsfw, NULL, NULL, NULL, NULL, (int32_t*)dst, s));
  mxg_operand_t A = {dqx, (const uint8_t*)dsfx, NULL};
  mxg_operand_t B = {dqw, (const uint8_t*)dsfw, NULL};
  MK(mxg_grouped_gemm(MXG_MXFP8_E4M3, MXG_FPROP_TN, &A, &B, (const int64_t*)dws, G, M, N, K, NULL,
                      NULL, NULL, dc, MXG_OUT_F32, NULL, 0, (int32_t*)dst, s));
  CK(cudaStreamSynchronize(stream));
  CK(cudaMemcpy(hc, dc, (size_t)M * N * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&hst, dst, 4, cudaMemcpyDeviceToHost));
  if (hst != 0) {
    fprintf(stderr, "device status %d\n", hst);
    return 4;
  }
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      const int g = m / 128;
      const float want = (float)((n + 3 * (m % 128) + 5 * g) % 9 - 4);
      if (hc[(size_t)m * N + n] != want) {
        fprintf(stderr, "C[%d,%d] = %g, expected %g\n", m, n, hc[(size_t)m * N + n], want);
        return 5;
      }
    }
  printf("c_abi_example ok: %llu launches\n", (unsigned long long)mxg_launch_count());
  return 0;
}
