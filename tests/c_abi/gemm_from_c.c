/*
 * A plain C caller of the GEMM C ABI (include/gb300_gemm.h): no Python, no torch.  It owns
 * its device buffers (CUDA runtime), calls gb_gemm_f16 on a stream with a K-major A and an
 * MN-major B, reads the device status word, and checks D exactly: the operands are small
 * integers, so every sum is an integer far below 2^11 and exact in fp16 and fp32.  Then it
 * calls gb_gemm_f16_host with plain malloc'd (pageable) host buffers: the same problem
 * (D must equal the device call's bit for bit), and a taller one with an M-major A that the
 * library stages in four row blocks, checked exactly against integer sums.
 * Exit status 0 on success.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "gb300_gemm.h"

static uint16_t f16_of_int(int v) {
  /* exact binary16 encoding of a small integer (|v| < 2048) */
  if (v == 0) return 0;
  uint16_t sign = v < 0 ? 0x8000u : 0u;
  unsigned a = (unsigned)(v < 0 ? -v : v);
  int e = 0;
  while ((a >> e) > 1) ++e;
  unsigned frac = (a << (10 - e)) & 0x3FFu;
  return (uint16_t)(sign | ((unsigned)(e + 15) << 10) | frac);
}

static int int_of_f16(uint16_t h) {
  int e = (h >> 10) & 0x1F, f = h & 0x3FF;
  if (e == 0) return 0; /* only exact small integers are expected */
  int mag = (1 << 10 | f);
  mag = e - 25 >= 0 ? mag << (e - 25) : mag >> (25 - e);
  return (h & 0x8000u) ? -mag : mag;
}

int main(void) {
  const int64_t M = 300, N = 200, K = 136, lda = 136, ldb = 200; /* A K-major, B N-major */
  uint16_t *A = malloc(M * lda * 2), *B = malloc(K * ldb * 2), *C = malloc(M * N * 2), *D = malloc(M * N * 2);
  int *a = malloc(M * K * sizeof(int)), *b = malloc(K * N * sizeof(int)), *c = malloc(M * N * sizeof(int));
  if (!A || !B || !C || !D || !a || !b || !c) return 2;
  unsigned s = 12345u;
  for (int64_t i = 0; i < M * K; ++i) { s = s * 1103515245u + 12345u; a[i] = (int)((s >> 16) % 5) - 2; }
  for (int64_t i = 0; i < K * N; ++i) { s = s * 1103515245u + 12345u; b[i] = (int)((s >> 16) % 5) - 2; }
  for (int64_t i = 0; i < M * N; ++i) { s = s * 1103515245u + 12345u; c[i] = (int)((s >> 16) % 5) - 2; }
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) A[m * lda + k] = f16_of_int(a[m * K + k]);
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n) B[k * ldb + n] = f16_of_int(b[k * N + n]);
  for (int64_t i = 0; i < M * N; ++i) C[i] = f16_of_int(c[i]);

  void *dA, *dB, *dC, *dD;
  cudaStream_t st;
  if (cudaMalloc(&dA, M * lda * 2) || cudaMalloc(&dB, K * ldb * 2) || cudaMalloc(&dC, M * N * 2) ||
      cudaMalloc(&dD, M * N * 2) || cudaStreamCreate(&st))
    return 3;
  cudaMemcpy(dA, A, M * lda * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, B, K * ldb * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dC, C, M * N * 2, cudaMemcpyHostToDevice);
  gb_status r = gb_gemm_f16(M, N, K, 1.0f, dA, lda, GB_K_MAJOR, dB, ldb, GB_MN_MAJOR, 1.0f, dC, dD, st);
  if (r != GB_OK) { fprintf(stderr, "gb_gemm_f16: %s\n", gb_status_string(r)); return 4; }
  uint32_t detail = 0;
  r = gb_last_device_status(st, &detail);
  if (r != GB_OK) { fprintf(stderr, "device status: %s (%#x)\n", gb_status_string(r), detail); return 5; }
  cudaMemcpy(D, dD, M * N * 2, cudaMemcpyDeviceToHost);
  long bad = 0;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int want = c[m * N + n];
      for (int64_t k = 0; k < K; ++k) want += a[m * K + k] * b[k * N + n];
      if (int_of_f16(D[m * N + n]) != want) ++bad;
    }
  /* argument errors come back before any launch */
  if (gb_gemm_f16(M, N, K, 1.0f, (char*)dA + 2, lda, GB_K_MAJOR, dB, ldb, GB_MN_MAJOR, 0.0f, NULL, dD, st) !=
      GB_ERR_MISALIGNED)
    return 6;
  if (gb_gemm_f16(M, N, K, 1.0f, dA, lda, GB_K_MAJOR, dB, ldb, GB_MN_MAJOR, 1.0f, NULL, dD, st) != GB_ERR_INVALID_ARG)
    return 7;
  printf("C ABI: %ld of %ld outputs wrong\n", bad, (long)(M * N));

  /* host buffers: the same problem through gb_gemm_f16_host */
  uint16_t* D2 = malloc(M * N * 2);
  if (!D2) return 2;
  r = gb_gemm_f16_host(M, N, K, 1.0f, A, lda, GB_K_MAJOR, B, ldb, GB_MN_MAJOR, 1.0f, C, D2, st);
  if (r != GB_OK) { fprintf(stderr, "gb_gemm_f16_host: %s\n", gb_status_string(r)); return 8; }
  if (cudaStreamSynchronize(st) != cudaSuccess) return 9;
  long diff = 0;
  for (int64_t i = 0; i < M * N; ++i) diff += D2[i] != D[i];
  printf("host call: %ld of %ld outputs differ from the device call\n", diff, (long)(M * N));
  /* device pointers are refused by the host entry point */
  if (gb_gemm_f16_host(M, N, K, 1.0f, dA, lda, GB_K_MAJOR, dB, ldb, GB_MN_MAJOR, 0.0f, NULL, D2, st) !=
      GB_ERR_INVALID_ARG)
    return 10;

  /* a taller problem, M-major A (column-major, lda >= M2), staged in row blocks */
  const int64_t M2 = 4352, lda2 = 4360;
  int64_t bounds[9];
  int nblocks = 0;
  if (gb_gemm_host_row_blocks(M2, bounds, &nblocks) != GB_OK || nblocks != 4) return 11;
  uint16_t *A2 = malloc(K * lda2 * 2), *C2 = malloc(M2 * N * 2), *D3 = malloc(M2 * N * 2);
  int *a2 = malloc(M2 * K * sizeof(int)), *c2 = malloc(M2 * N * sizeof(int));
  if (!A2 || !C2 || !D3 || !a2 || !c2) return 2;
  for (int64_t i = 0; i < M2 * K; ++i) { s = s * 1103515245u + 12345u; a2[i] = (int)((s >> 16) % 5) - 2; }
  for (int64_t i = 0; i < M2 * N; ++i) { s = s * 1103515245u + 12345u; c2[i] = (int)((s >> 16) % 5) - 2; }
  for (int64_t k = 0; k < K; ++k)
    for (int64_t m = 0; m < M2; ++m) A2[m + k * lda2] = f16_of_int(a2[m * K + k]);
  for (int64_t i = 0; i < M2 * N; ++i) C2[i] = f16_of_int(c2[i]);
  r = gb_gemm_f16_host(M2, N, K, 1.0f, A2, lda2, GB_MN_MAJOR, B, ldb, GB_MN_MAJOR, -1.0f, C2, D3, st);
  if (r != GB_OK) { fprintf(stderr, "gb_gemm_f16_host (M-major): %s\n", gb_status_string(r)); return 12; }
  if (cudaStreamSynchronize(st) != cudaSuccess) return 13;
  long bad2 = 0;
  for (int64_t m = 0; m < M2; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int want = -c2[m * N + n];
      for (int64_t k = 0; k < K; ++k) want += a2[m * K + k] * b[k * N + n];
      if (int_of_f16(D3[m * N + n]) != want) ++bad2;
    }
  printf("host call, M-major A in %d row blocks: %ld of %ld outputs wrong\n", nblocks, bad2, (long)(M2 * N));
  if (gb_host_staging_free() != GB_OK) return 14;
  cudaFree(dA); cudaFree(dB); cudaFree(dC); cudaFree(dD); cudaStreamDestroy(st);
  return (bad == 0 && diff == 0 && bad2 == 0) ? 0 : 1;
}
