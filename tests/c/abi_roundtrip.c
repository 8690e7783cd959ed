/* Plain-C use of the zpp ABI (no Python, no torch): quantise two hand-derived blocks,
 * check codes, scales and the dequantised values, then exercise the error paths.
 * Expected values: tests/golden/quant_tiny.txt, case int4_ties, each 4-element block
 * embedded at the start of a 64-element block of zeros (zeros leave absmax, scale and
 * codes unchanged). Then qgZ step 1 on the same data, flat and as a list of two tensors.
 * Exit status 0 on success. */
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

  /* qgZ step 1 on one rank (topology 1 x 1), once on the flat buffer and once with the same
   * 128 elements given as two tensors of 64 (host arrays of device pointers and sizes):
   * the outputs must be identical. */
  {
    const zpp_topology one = {1, 1};
    void *dc1 = NULL, *dc2 = NULL;
    float *ds1 = NULL, *ds2 = NULL;
    CHECK(cudaMalloc(&dc1, N / 2) == cudaSuccess && cudaMalloc(&dc2, N / 2) == cudaSuccess, "cudaMalloc c");
    CHECK(cudaMalloc((void**)&ds1, NB * sizeof(float)) == cudaSuccess, "cudaMalloc s1");
    CHECK(cudaMalloc((void**)&ds2, NB * sizeof(float)) == cudaSuccess, "cudaMalloc s2");
    const void* tensors[2] = {dx, (const char*)dx + B * sizeof(unsigned short)};
    const int64_t sizes[2] = {B, B};
    CHECK(zpp_qgz_reorder_quant(dx, ZPP_F16, N, B, 4, one, dc1, ds1, 0) == ZPP_OK, "flat step 1");
    CHECK(zpp_qgz_reorder_quant_tensors(tensors, sizes, 2, ZPP_F16, B, 4, one, dc2, ds2, 0) == ZPP_OK,
          "tensor-list step 1");
    unsigned char c1[N / 2], c2[N / 2];
    float s1[NB], s2[NB];
    CHECK(cudaMemcpy(c1, dc1, sizeof c1, cudaMemcpyDeviceToHost) == cudaSuccess, "copy c1");
    CHECK(cudaMemcpy(c2, dc2, sizeof c2, cudaMemcpyDeviceToHost) == cudaSuccess, "copy c2");
    CHECK(cudaMemcpy(s1, ds1, sizeof s1, cudaMemcpyDeviceToHost) == cudaSuccess, "copy s1");
    CHECK(cudaMemcpy(s2, ds2, sizeof s2, cudaMemcpyDeviceToHost) == cudaSuccess, "copy s2");
    CHECK(memcmp(c1, c2, sizeof c1) == 0 && memcmp(s1, s2, sizeof s1) == 0, "tensor list == flat");
    const int64_t odd[2] = {B + 8, B - 8};
    CHECK(zpp_qgz_reorder_quant_tensors(tensors, odd, 2, ZPP_F16, B, 4, one, dc2, ds2, 0) ==
              ZPP_ERR_MISALIGNED, "tensor sizes must be multiples of 16");
    cudaFree(dc1);
    cudaFree(dc2);
    cudaFree(ds1);
    cudaFree(ds2);
  }

  /* rejected before any launch; nothing written */
  CHECK(zpp_quant_blockwise(dx, ZPP_F16, N, 100, 4, dcodes, dscales, 0) == ZPP_ERR_INVALID_ARG, "bad block");
  CHECK(zpp_quant_blockwise(dx, ZPP_F16, N, B, 3, dcodes, dscales, 0) == ZPP_ERR_INVALID_ARG, "bad bits");
  CHECK(zpp_quant_blockwise((char*)dx + 8, ZPP_F16, 64, B, 4, dcodes, dscales, 0) == ZPP_ERR_MISALIGNED, "misaligned");
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
