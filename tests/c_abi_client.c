/* A plain C client of include/nvfp4.h: no PyTorch, only the CUDA runtime.
 * It builds a deterministic bf16 tensor on the host, quantizes it with every
 * scale rule through nvfp4_quantize, dequantizes, and prints, per rule, alpha
 * and FNV-1a hashes of the codes, the scales and the dequantized tensor, so
 * that a test can compare them with the same calls made through the Python
 * binding.  Usage: c_abi_client ROWS COLS */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "nvfp4.h"

static uint64_t fnv1a(const uint8_t *p, size_t n) {
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

/* bf16 bits of element i: a fixed integer recipe (xorshift), magnitudes up to ~0.1 */
static uint16_t weight_bits(uint64_t i) {
  uint64_t x = i * 0x9E3779B97F4A7C15ull + 12345u;
  x ^= x >> 33;
  x *= 0xFF51AFD7ED558CCDull;
  x ^= x >> 33;
  uint16_t sign = (uint16_t)((x >> 8) & 0x8000u);
  uint16_t exp = (uint16_t)(113u + (x % 11u));  /* 2^-14 .. 2^-4 */
  uint16_t man = (uint16_t)((x >> 20) & 0x7Fu);
  return (uint16_t)(sign | (exp << 7) | man);
}

#define CHECK(call)                                                        \
  do {                                                                     \
    int rc_ = (int)(call);                                                 \
    if (rc_ != 0) {                                                        \
      fprintf(stderr, "%s failed: %d\n", #call, rc_);                    \
      return 1;                                                            \
    }                                                                      \
  } while (0)

int main(int argc, char **argv) {
  if (argc != 3) return 2;
  const int64_t rows = atoll(argv[1]), cols = atoll(argv[2]);
  const size_t n = (size_t)(rows * cols);
  uint16_t *w = (uint16_t *)malloc(n * 2);
  uint8_t *codes = (uint8_t *)malloc(n / 2), *scales = (uint8_t *)malloc(n / 16);
  uint16_t *deq = (uint16_t *)malloc(n * 2);
  if (!w || !codes || !scales || !deq) return 3;
  for (size_t i = 0; i < n; ++i) w[i] = weight_bits(i);
  void *dW, *dC, *dS, *dA, *dD;
  CHECK(cudaMalloc(&dW, n * 2));
  CHECK(cudaMalloc(&dC, n / 2));
  CHECK(cudaMalloc(&dS, n / 16));
  CHECK(cudaMalloc(&dA, 4));
  CHECK(cudaMalloc(&dD, n * 2));
  CHECK(cudaMemcpy(dW, w, n * 2, cudaMemcpyHostToDevice));
  cudaStream_t st;
  CHECK(cudaStreamCreate(&st));
  for (int mode = 0; mode <= 3; ++mode) {
    const int iters = mode >= 2 ? 3 : 0;
    CHECK(nvfp4_quantize(dW, rows, cols, mode, iters, (uint8_t *)dC, (uint8_t *)dS, (float *)dA, st));
    CHECK(nvfp4_dequantize((const uint8_t *)dC, (const uint8_t *)dS, (const float *)dA, rows, cols, dD, st));
    CHECK(cudaStreamSynchronize(st));
    float alpha;
    CHECK(cudaMemcpy(&alpha, dA, 4, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(codes, dC, n / 2, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(scales, dS, n / 16, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(deq, dD, n * 2, cudaMemcpyDeviceToHost));
    uint32_t abits;
    memcpy(&abits, &alpha, 4);
    printf("%d %08x %016llx %016llx %016llx\n", mode, abits, (unsigned long long)fnv1a(codes, n / 2),
           (unsigned long long)fnv1a(scales, n / 16), (unsigned long long)fnv1a((const uint8_t *)deq, n * 2));
  }
  printf("%s\n", nvfp4_status_string(NVFP4_ERR_MISALIGNED));
  cudaStreamDestroy(st);
  cudaFree(dW);
  cudaFree(dC);
  cudaFree(dS);
  cudaFree(dA);
  cudaFree(dD);
  free(w);
  free(codes);
  free(scales);
  free(deq);
  return 0;
}
