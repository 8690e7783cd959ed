// reorder_tensors_bf16.cu -- K3T (reorder_tensors.cuh) for bf16 gradients.
#include "reorder_tensors.cuh"

namespace zpp {

cudaError_t launch_reorder_quant_tensors_bf16(const TensorTable& tab, int64_t E, int block,
                                              int bits, int N, int M, bool v8, void* codes,
                                              float* scales, cudaStream_t s) {
  return run_reorder_quant_tensors<BF16>(tab, E, block, bits, N, M, v8, codes, scales, s);
}

}  // namespace zpp
