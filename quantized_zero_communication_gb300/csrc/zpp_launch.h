// zpp_launch.h -- host-side launchers of the sm_103a kernels (internal to libzpp).
// The C ABI in zpp_abi.cu validates arguments and then calls exactly one of these.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

namespace zpp {

// K1: block quantisation of n fp16 (is_bf16 = 0) or bf16 values.
cudaError_t launch_quant(const void* x, int is_bf16, int64_t n, int block, int bits,
                         void* codes, float* scales, cudaStream_t s);

// K2: dequantisation into fp16 (out_kind 0), bf16 (1) or fp32 (2).
cudaError_t launch_dequant(const void* codes, const float* scales, int64_t n, int block,
                           int bits, void* y, int out_kind, cudaStream_t s);

// The qgZ launchers cover the hop-1 chunks / receivers with local index l in
// [l_begin, l_end) (the whole exchange is [0, M)).
// K3: slice reorder + block quantisation of `ranks` consecutive ranks of E elements each
// (all W = N*M ranks of the virtual layout, or the one rank of a real device).
cudaError_t launch_reorder_quant(const void* grads, int is_bf16, int64_t E, int block, int bits,
                                 int N, int M, int l_begin, int l_end, int ranks, void* codes,
                                 float* scales, cudaStream_t s);

// K3 over a bucket given as tensors (the flatten fused in; whole exchange only). Tensor t
// holds the W ranks' copies back to back, rank r's at ptr[t] + r * len_t, len_t =
// offs[t+1] - offs[t]; offs[0] = 0, offs[count] = E. Passed by value in the kernel's
// parameter space (about 16 KB), so no device table is needed.
constexpr int kMaxTensors = 1024;  // = ZPP_MAX_TENSORS
struct TensorTable {
  const uint16_t* ptr[kMaxTensors];
  int64_t offs[kMaxTensors + 1];
  int32_t count;
};
cudaError_t launch_reorder_quant_tensors(const TensorTable& tab, int is_bf16, int64_t E, int block,
                                         int bits, int N, int M, void* codes, float* scales,
                                         cudaStream_t s);
// The same per input type (v8: every tensor pointer is 32-byte aligned).
cudaError_t launch_reorder_quant_tensors_f16(const TensorTable& tab, int64_t E, int block,
                                             int bits, int N, int M, bool v8, void* codes,
                                             float* scales, cudaStream_t s);
cudaError_t launch_reorder_quant_tensors_bf16(const TensorTable& tab, int64_t E, int block,
                                              int bits, int N, int M, bool v8, void* codes,
                                              float* scales, cudaStream_t s);

// K4: intra-node fused dequantise -> fp32 sum over M sources -> requantise. Receiver
// (n, l), n < N, reads C elements at offset l*C of sources n*M .. n*M+M-1, which lie E
// elements apart, and writes C codes at receiver offset (n*M + l)*C. The virtual layout
// has C = E / M; one real rank's received chunks are N = 1, l = 0 and E = C.
cudaError_t launch_dequant_reduce_requant(const void* codes, const float* scales, int64_t E,
                                          int64_t C, int block, int bits, int N, int M,
                                          int l_begin, int l_end, void* out_codes,
                                          float* out_scales, cudaStream_t s);

// K5: inter-node dequantise -> fp32 sum over N slices, times post_scale, stored as fp16
// (out_kind 0), bf16 (1) or fp32 (2). Receiver (n, l), n < nz, reads S elements at offset
// n*S of the N hop-1 outputs of ranks (n', l), which are C elements long and M outputs
// apart, and writes S outputs at (n*M + l)*S. The virtual layout has S = E / W, C = E / M,
// nz = N; one real rank's received slices are S = C, M = 1, nz = 1, l = 0.
cudaError_t launch_dequant_reduce(const void* codes, const float* scales, int64_t S, int64_t C,
                                  int block, int bits, int N, int M, int l_begin, int l_end,
                                  int nz, float post_scale, void* out, int out_kind,
                                  cudaStream_t s);

// The device fault word: bits set by kernels whose bounded waits ran out (1: a producer
// wait of the INT8 K4 ring, 2: a consumer wait of that ring, 4: the wait self-test).
// Synchronous: copies the word of the current device to *flags, then zeroes it if clear.
cudaError_t read_device_fault(unsigned* flags, bool clear);

// A kernel that waits, bounded by limit_ns, on a barrier nothing completes (sets bit 4).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);

// K6: 256-bit device copy (the same-run HBM reference).
cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, cudaStream_t s);

// Grid size when every CTA owns `per_cta` consecutive tiles and exits (no grid-stride
// loop): on GB300 a streaming kernel launched this way sustains more HBM bandwidth than
// a persistent grid sized to the SM count.
inline int tile_grid(int64_t tiles, int per_cta) {
  int64_t g = (tiles + per_cta - 1) / per_cta;
  return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace zpp
