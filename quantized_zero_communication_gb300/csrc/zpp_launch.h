// zpp_launch.h -- host-side launchers of the sm_103a kernels (internal to libzpp).
// The C ABI in zpp_abi.cu validates arguments and then calls exactly one of these.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

namespace zpp {

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// K1: block quantisation of n fp16 (is_bf16 = 0) or bf16 values.
cudaError_t launch_quant(const void* x, int is_bf16, int64_t n, int block, int bits,
                         void* codes, float* scales, cudaStream_t s);

// K2: dequantisation into fp16 (out_kind 0), bf16 (1) or fp32 (2).
cudaError_t launch_dequant(const void* codes, const float* scales, int64_t n, int block,
                           int bits, void* y, int out_kind, cudaStream_t s);

// K3: slice reorder + block quantisation of W = N*M ranks of E elements.
cudaError_t launch_reorder_quant(const void* grads, int is_bf16, int64_t E, int block,
                                 int bits, int N, int M, void* codes, float* scales,
                                 cudaStream_t s);

// K4: intra-node fused dequantise -> fp32 sum over M chunks -> requantise.
cudaError_t launch_dequant_reduce_requant(const void* codes, const float* scales, int64_t E,
                                          int block, int bits, int N, int M, void* out_codes,
                                          float* out_scales, cudaStream_t s);

// K5: inter-node dequantise -> fp32 sum over N slices.
cudaError_t launch_dequant_reduce(const void* codes, const float* scales, int64_t E, int block,
                                  int bits, int N, int M, float* out, cudaStream_t s);

// K6: 256-bit device copy (the same-run HBM reference).
cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, cudaStream_t s);

// Grid size for a persistent kernel: enough CTAs to fill every SM at the kernel's
// occupancy, never more than there is work for.
inline int persistent_grid(int64_t work_ctas, int ctas_per_sm) {
  int64_t full = static_cast<int64_t>(sm_count()) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  int64_t g = work_ctas < full ? work_ctas : full;
  return static_cast<int>(g > 0 ? g : 1);
}

template <typename Kernel>
int occupancy_of(Kernel k, int threads, size_t smem = 0) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace zpp
