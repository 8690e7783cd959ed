/* Plain-C use of the zpp ABI (no Python, no torch): quantise two hand-derived blocks,
 * check codes, scales and the dequantised values, then exercise the error paths.
 * Expected values: tests/golden/quant_tiny.txt, case int4_ties, each 4-element block
 * embedded at the start of a 64-element block of zeros (zeros leave absmax, scale and
 * codes unchanged). Exit status 0 on success. */
#include <stdio.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "zpp.h"

#define CHECK(cond, what)                      \
  do {                                         \
    if (!(cond)) {                             \
      fprintf(stderr, "FAILED: %s\n", what);   \
      return 1;                                \
    }                                          \
  } while (0)

static unsigned short f16_bits(float v) { /* exact for the small values used here */
  if (v == 0.0f) return 0;
  unsigned short s = v < 0 ? 0x8000 : 0;
  float a = v < 0 ? -v : v;
  int e = 0;
  while (a >= 2.0f) { a /= 2.0f; ++e; }
  while (a < 1.0f) { a *= 2.0f; --e; }
  return (unsigned short)(s | ((e + 15) << 10) | (unsigned short)((a - 1.0f) * 1024.0f));
}

int main(void) {
  const float x_blocks[2][4] = {{7, 0.5f, 1.5f, -2.5f}, {-14, 1, 3, 5}};
  const unsigned char want_codes[2][2] = {{0x07, 0xe2}, {0x09, 0x22}};
  const float want_scale[2] = {1.0f, 2.0f};
  const float want_y[2][4] = {{7, 0, 2, -2}, {-14, 0, 4, 4}};
  enum { B = 64, NB = 2, N = B * NB };
  unsigned short hx[N];
  memset(hx, 0, sizeof hx);
  for (int b = 0; b < NB; ++b)
    for (int i = 0; i < 4; ++i) hx[b * B + i] = f16_bits(x_blocks[b][i]);

  void *dx = NULL, *dcodes = NULL, *dy = NULL;
  float* dscales = NULL;
  CHECK(cudaMalloc(&dx, sizeof hx) == cudaSuccess, "cudaMalloc x");
  CHECK(cudaMalloc(&dcodes, N / 2) == cudaSuccess, "cudaMalloc codes");
  CHECK(cudaMalloc((void**)&dscales, NB * sizeof(float)) == cudaSuccess, "cudaMalloc scales");
  CHECK(cudaMalloc(&dy, N * sizeof(float)) == cudaSuccess, "cudaMalloc y");
  CHECK(cudaMemcpy(dx, hx, sizeof hx, cudaMemcpyHostToDevice) == cudaSuccess, "copy in");

  CHECK(zpp_quant_blockwise(dx, ZPP_F16, N, B, 4, dcodes, dscales, 0) == ZPP_OK, "quant");
  CHECK(zpp_dequant_blockwise(dcodes, dscales, N, B, 4, dy, ZPP_F32, 0) == ZPP_OK, "dequant");
  unsigned char codes[N / 2];
  float scales[NB], y[N];
  CHECK(cudaMemcpy(codes, dcodes, sizeof codes, cudaMemcpyDeviceToHost) == cudaSuccess, "copy codes");
  CHECK(cudaMemcpy(scales, dscales, sizeof scales, cudaMemcpyDeviceToHost) == cudaSuccess, "copy scales");
  CHECK(cudaMemcpy(y, dy, sizeof y, cudaMemcpyDeviceToHost) == cudaSuccess, "copy y");
  for (int b = 0; b < NB; ++b) {
    CHECK(codes[b * B / 2] == want_codes[b][0] && codes[b * B / 2 + 1] == want_codes[b][1], "codes");
    CHECK(scales[b] == want_scale[b], "scales");
    for (int i = 0; i < 4; ++i) CHECK(y[b * B + i] == want_y[b][i], "dequantised values");
    for (int i = 4; i < B; ++i) CHECK(y[b * B + i] == 0.0f, "zero padding");
  }

  /* rejected before any launch; nothing written */
  CHECK(zpp_quant_blockwise(dx, ZPP_F16, N, 100, 4, dcodes, dscales, 0) == ZPP_ERR_INVALID_ARG, "bad block");
  CHECK(zpp_quant_blockwise(dx, ZPP_F16, N, B, 3, dcodes, dscales, 0) == ZPP_ERR_INVALID_ARG, "bad bits");
  CHECK(zpp_quant_blockwise((char*)dx + 16, ZPP_F16, 64, B, 4, dcodes, dscales, 0) == ZPP_ERR_MISALIGNED, "misaligned");
  CHECK(zpp_code_bytes(7, 4) == 4 && zpp_num_scales(1000, 256) == 4, "size helpers");
  CHECK(strncmp(zpp_status_string(ZPP_ERR_MISALIGNED), "ZPP_ERR_MISALIGNED", 18) == 0, "status string");
  CHECK(cudaDeviceSynchronize() == cudaSuccess, "device sync");
  cudaFree(dx);
  cudaFree(dcodes);
  cudaFree(dscales);
  cudaFree(dy);
  printf("zpp C ABI round trip OK\n");
  return 0;
}
