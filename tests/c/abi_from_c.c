/*
 * abi_from_c.c -- the C ABI of libnf4 used from plain C (no Python, no torch).
 *
 * Test program, built and run by tests/test_abi.py (no GPU: argument checks,
 * the codebook, workspace sizes) and tests/test_zzz_c_abi_gpu.py (GPU: the
 * down projection with its residual, dumped for comparison with the oracle).
 *
 *   abi_from_c            host-side checks only; exit 0 on success
 *   abi_from_c OUT.bin    host-side checks, then, if a CUDA device is present,
 *                         quantize a seeded 2048 x 11008 weight on the device,
 *                         run nf4_gemv_residual with bf16 x, and write
 *                         W (fp32), x (bf16 bits), r, codes, scales, y to OUT.bin
 *
 * Every failure prints a line and exits non-zero.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "nf4.h"

#define CHECK(cond, ...)                 \
  do {                                   \
    if (!(cond)) {                       \
      fprintf(stderr, "FAIL: " __VA_ARGS__); \
      fprintf(stderr, "\n");             \
      exit(1);                           \
    }                                    \
  } while (0)

/* splitmix64: a seeded stream of 64-bit values (inputs only, no method arithmetic) */
static uint64_t g_state;
static uint64_t next_u64(void) {
  uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
/* uniform in [-1, 1) with 24 random bits, exact in fp32 */
static float next_unit(void) { return (float)((int64_t)(next_u64() >> 40) - (1 << 23)) / (float)(1 << 23); }

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static void host_checks(void) {
  float cb[16];
  nf4_codebook(cb);
  CHECK(cb[0] == -1.0f && cb[7] == 0.0f && cb[15] == 1.0f, "codebook ends and zero level");
  for (int i = 0; i < 15; ++i) CHECK(cb[i] < cb[i + 1], "codebook not increasing at %d", i);

  /* arguments are checked before anything touches a device */
  nf4_weight w = {(const uint8_t*)(uintptr_t)4096, (const float*)(uintptr_t)4096, 8, 100};
  CHECK(nf4_gemv(&w, (const void*)(uintptr_t)4096, NF4_BF16, (float*)(uintptr_t)4096, NULL) == NF4_EINVAL,
        "K = 100 accepted");
  CHECK(strlen(nf4_last_error()) > 0, "no message for a failed call");
  w.K = 128;
  CHECK(nf4_gemv(&w, NULL, NF4_BF16, (float*)(uintptr_t)4096, NULL) == NF4_ENULL, "NULL x accepted");
  CHECK(nf4_gemv(NULL, (const void*)(uintptr_t)4096, NF4_BF16, (float*)(uintptr_t)4096, NULL) == NF4_ENULL,
        "NULL weight accepted");
  w.codes = (const uint8_t*)(uintptr_t)4097;
  CHECK(nf4_gemv(&w, (const void*)(uintptr_t)4096, NF4_BF16, (float*)(uintptr_t)4096, NULL) == NF4_EALIGN,
        "unaligned codes accepted");
  CHECK(nf4_workspace_bytes(151936, 2048, 1) >= 16, "argmax workspace");
  CHECK(strstr(nf4_describe_launch("transpose", 8, 128, 1), "invalid operation") != NULL, "unknown op described");
  CHECK(strstr(nf4_describe_launch("residual", 8, 100, 1), "invalid shape") != NULL, "K = 100 described");
  printf("host checks ok\n");
}

#define CUDA_OK(call)                                                           \
  do {                                                                          \
    cudaError_t e_ = (call);                                                    \
    CHECK(e_ == cudaSuccess, "%s: %s", #call, cudaGetErrorString(e_));          \
  } while (0)

static void write_all(FILE* f, const void* p, size_t n) { CHECK(fwrite(p, 1, n, f) == n, "short write"); }

static void device_run(const char* path) {
  const int64_t M = 2048, K = 11008;
  const size_t nw = (size_t)(M * K);
  float* W = (float*)malloc(nw * 4);
  uint16_t* x = (uint16_t*)malloc((size_t)K * 2);
  float* r = (float*)malloc((size_t)M * 4);
  uint8_t* codes = (uint8_t*)malloc(nw / 2);
  float* scales = (float*)malloc(nw / 64 * 4);
  float* y = (float*)malloc((size_t)M * 4);
  CHECK(W && x && r && codes && scales && y, "host allocation");
  g_state = 20251;
  for (size_t i = 0; i < nw; ++i) W[i] = 0.02f * next_unit();
  for (int64_t k = 0; k < K; ++k) x[k] = f32_to_bf16_rne(next_unit());
  for (int64_t m = 0; m < M; ++m) r[m] = next_unit();

  float *dW, *dr, *dy, *dscales;
  uint16_t* dx;
  uint8_t* dcodes;
  CUDA_OK(cudaMalloc((void**)&dW, nw * 4));
  CUDA_OK(cudaMalloc((void**)&dx, (size_t)K * 2));
  CUDA_OK(cudaMalloc((void**)&dr, (size_t)M * 4));
  CUDA_OK(cudaMalloc((void**)&dy, (size_t)M * 4));
  CUDA_OK(cudaMalloc((void**)&dcodes, nw / 2));
  CUDA_OK(cudaMalloc((void**)&dscales, nw / 64 * 4));
  CUDA_OK(cudaMemcpy(dW, W, nw * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dx, x, (size_t)K * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dr, r, (size_t)M * 4, cudaMemcpyHostToDevice));

  nf4_status st = nf4_quantize(dW, M, K, dcodes, dscales, NULL);
  CHECK(st == NF4_OK, "nf4_quantize: %d %s", (int)st, nf4_last_error());
  nf4_weight w = {dcodes, dscales, M, K};
  st = nf4_gemv_residual(&w, dx, NF4_BF16, dr, dy, NULL);
  CHECK(st == NF4_OK, "nf4_gemv_residual: %d %s", (int)st, nf4_last_error());
  CUDA_OK(cudaDeviceSynchronize());
  CHECK(nf4_check_device_errors() == NF4_OK, "device error word set");
  CUDA_OK(cudaMemcpy(codes, dcodes, nw / 2, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(scales, dscales, nw / 64 * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(y, dy, (size_t)M * 4, cudaMemcpyDeviceToHost));

  FILE* f = fopen(path, "wb");
  CHECK(f != NULL, "cannot open %s", path);
  write_all(f, W, nw * 4);
  write_all(f, x, (size_t)K * 2);
  write_all(f, r, (size_t)M * 4);
  write_all(f, codes, nw / 2);
  write_all(f, scales, nw / 64 * 4);
  write_all(f, y, (size_t)M * 4);
  CHECK(fclose(f) == 0, "close %s", path);
  cudaFree(dW);
  cudaFree(dx);
  cudaFree(dr);
  cudaFree(dy);
  cudaFree(dcodes);
  cudaFree(dscales);
  free(W);
  free(x);
  free(r);
  free(codes);
  free(scales);
  free(y);
  printf("device run ok\n");
}

int main(int argc, char** argv) {
  host_checks();
  if (argc < 2) return 0;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    printf("no CUDA device\n");
    return 0;
  }
  device_run(argv[1]);
  return 0;
}
