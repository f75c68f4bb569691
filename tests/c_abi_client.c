/* A plain C client of the library: grouped NVFP4 GEMM through the C ABI with a
 * closed-form answer, plus the documented argument errors.  Built and run by
 * tests/test_gpu_c_client.py.
 *
 * Every A code byte is 0x22 (two E2M1 codes of 1.0: exponent field 1,
 * mantissa 0), every scale byte 0x38 (E4M3 1.0: exponent field 7), and B is
 * 0x22 for group 0 and 0xAA (E2M1 -1.0, sign bit set) for group 1, so each
 * product in the K sum is +1 or -1 and C = +K or -K exactly in fp16. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "nvfp4_gemm.h"

#define CHECK(cond, ...)                \
  do {                                  \
    if (!(cond)) {                      \
      fprintf(stderr, __VA_ARGS__);     \
      fprintf(stderr, "\n");            \
      return 1;                         \
    }                                   \
  } while (0)

/* fp16 bit pattern of +/-K for K a power of two up to 2^15 */
static uint16_t half_of_pow2(int k, int negative) {
  int e = 0;
  while ((1 << e) < k) ++e;
  return (uint16_t)(((negative ? 1u : 0u) << 15) | ((uint32_t)(e + 15) << 10));
}

int main(void) {
  enum { G = 2 };
  const int M[G] = {200, 128}, N[G] = {264, 1024}, K[G] = {512, 1024}, L[G] = {1, 2};
  const unsigned char bcode[G] = {0x22, 0xAA};
  void *A[G], *B[G], *SFAraw[G], *SFBraw[G], *SFA[G], *SFB[G], *C[G];
  for (int g = 0; g < G; ++g) {
    const size_t a = (size_t)L[g] * M[g] * K[g] / 2, b = (size_t)L[g] * N[g] * K[g] / 2;
    const size_t sa = (size_t)L[g] * M[g] * K[g] / 16, sb = (size_t)L[g] * N[g] * K[g] / 16;
    const size_t ra = nvfp4_gemm_repacked_scales_bytes(M[g], K[g], L[g]);
    const size_t rb = nvfp4_gemm_repacked_scales_bytes(N[g], K[g], L[g]);
    CHECK(ra > 0 && rb > 0, "repacked size");
    CHECK(cudaMalloc(&A[g], a) == cudaSuccess && cudaMalloc(&B[g], b) == cudaSuccess &&
              cudaMalloc(&SFAraw[g], sa) == cudaSuccess && cudaMalloc(&SFBraw[g], sb) == cudaSuccess &&
              cudaMalloc(&SFA[g], ra) == cudaSuccess && cudaMalloc(&SFB[g], rb) == cudaSuccess &&
              cudaMalloc(&C[g], (size_t)L[g] * M[g] * N[g] * 2) == cudaSuccess,
          "cudaMalloc");
    cudaMemset(A[g], 0x22, a);
    cudaMemset(B[g], bcode[g], b);
    cudaMemset(SFAraw[g], 0x38, sa);
    cudaMemset(SFBraw[g], 0x38, sb);
    cudaMemset(C[g], 0xFF, (size_t)L[g] * M[g] * N[g] * 2);
    CHECK(nvfp4_gemm_repack_scales(SFAraw[g], SFA[g], M[g], K[g], L[g], NULL) == NVFP4_OK, "repack A: %s",
          nvfp4_gemm_last_error_string());
    CHECK(nvfp4_gemm_repack_scales(SFBraw[g], SFB[g], N[g], K[g], L[g], NULL) == NVFP4_OK, "repack B: %s",
          nvfp4_gemm_last_error_string());
  }
  int rc = nvfp4_gemm_run_grouped(G, (const void* const*)A, (const void* const*)B, (const void* const*)SFA,
                                  (const void* const*)SFB, C, M, N, K, L, NULL);
  CHECK(rc == NVFP4_OK, "run_grouped: %d %s", rc, nvfp4_gemm_last_error_string());
  CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
  CHECK(nvfp4_gemm_check_device_status(NULL) == NVFP4_OK, "device status");
  for (int g = 0; g < G; ++g) {
    const size_t n = (size_t)L[g] * M[g] * N[g];
    static uint16_t h[2 * 128 * 1024];
    CHECK(n <= sizeof h / 2, "buffer");
    CHECK(cudaMemcpy(h, C[g], n * 2, cudaMemcpyDeviceToHost) == cudaSuccess, "copy back");
    const uint16_t want = half_of_pow2(K[g], g == 1);
    for (size_t i = 0; i < n; ++i)
      CHECK(h[i] == want, "group %d element %zu: 0x%04x, want 0x%04x", g, i, h[i], want);
  }
  /* documented argument errors; nothing is launched */
  CHECK(nvfp4_gemm_run(NULL, B[0], SFA[0], SFB[0], C[0], M[0], N[0], K[0], 1, NULL) == NVFP4_ERR_INVALID_ARG,
        "null A");
  CHECK(strlen(nvfp4_gemm_last_error_string()) > 0, "error string");
  CHECK(nvfp4_gemm_run((char*)A[0] + 1, B[0], SFA[0], SFB[0], C[0], M[0], N[0], K[0], 1, NULL) ==
            NVFP4_ERR_INVALID_ARG,
        "misaligned A");
  CHECK(nvfp4_gemm_run(A[0], B[0], SFA[0], SFB[0], C[0], M[0], N[0], 100, 1, NULL) == NVFP4_ERR_UNSUPPORTED_SHAPE,
        "K %% 64");
  CHECK(nvfp4_gemm_run(A[0], B[0], SFA[0], SFB[0], C[0], M[0], 260, K[0], 1, NULL) == NVFP4_ERR_UNSUPPORTED_SHAPE,
        "N %% 8");
  CHECK(nvfp4_gemm_run_grouped(NVFP4_MAX_GROUPS + 1, (const void* const*)A, (const void* const*)B,
                               (const void* const*)SFA, (const void* const*)SFB, C, M, N, K, L,
                               NULL) == NVFP4_ERR_INVALID_ARG,
        "too many groups");
  for (int g = 0; g < G; ++g) {
    cudaFree(A[g]); cudaFree(B[g]); cudaFree(SFAraw[g]); cudaFree(SFBraw[g]);
    cudaFree(SFA[g]); cudaFree(SFB[g]); cudaFree(C[g]);
  }
  printf("c abi ok\n");
  return 0;
}
