// reorder_quant.cu -- K3: qgZ slice reorder + block quantisation of every rank's gradient
// (the warp tile of quant_tile.cuh), and the dispatch of K3T (reorder_tensors.cuh).
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model
// Training" (atlas.scime.ai summary), Approach: INT4 gradients, tensor-slice reordering
// for correct placement.
#include "quant_tile.cuh"
#include "reorder_tensors.cuh"

namespace zpp {

// K3: per source rank r, output slice position p = l_d*N + n_d holds original slice
// j = n_d*M + l_d. Grid (tile group, p - p_begin, r): each warp owns one warp tile of
// slice p of rank r (the last tile of a slice may be short but always holds whole
// blocks). A launch may cover only the slices of some hop-1 chunks (p_begin = l_begin*N).
template <typename TT, int BITS, int B, bool V8>
__global__ void __launch_bounds__(kThreads) k_reorder_quant(const uint16_t* __restrict__ grads,
                                                            int64_t E, int N, int M, int p_begin,
                                                            uint8_t* __restrict__ codes,
                                                            float* __restrict__ scales) {
  constexpr int TILE = QuantTile<B>::TILE;
  const int lane = threadIdx.x & 31;
  const int64_t k = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
  const int p = p_begin + static_cast<int>(blockIdx.y), r = blockIdx.z;
  if (k * TILE < S) {
    const int l_d = p / N, n_d = p - l_d * N;
    const int64_t j = static_cast<int64_t>(n_d) * M + l_d;
    const int64_t in_off = r * E + j * S + k * TILE;
    const int64_t out_off = r * E + p * S + k * TILE;
    const int64_t rem = S - k * TILE;
    if (rem >= TILE)
      quant_tile<TT, BITS, B, true>(FlatSrc<V8>{grads + in_off}, codes + out_off * BITS / 8,
                                    scales + out_off / B, TILE, lane);
    else
      quant_tile<TT, BITS, B, false>(FlatSrc<V8>{grads + in_off}, codes + out_off * BITS / 8,
                                     scales + out_off / B, static_cast<int>(rem), lane);
  }
}

template <typename TT, int BITS, int B, bool V8>
static cudaError_t run_reorder_quant(const void* g, int64_t E, int N, int M, int l_begin, int l_end,
                                     int ranks, void* codes, float* scales, cudaStream_t s) {
  auto kern = k_reorder_quant<TT, BITS, B, V8>;
  const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
  const int64_t tps = (S + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
  // output slice positions of chunks l_begin .. l_end-1: p in [l_begin*N, l_end*N)
  const dim3 grid(tile_grid(tps, kWarps), static_cast<unsigned>((l_end - l_begin) * N),
                  static_cast<unsigned>(ranks));
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(g), E, N, M, l_begin * N,
                                 static_cast<uint8_t*>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_reorder_quant_tensors(const TensorTable& tab, int is_bf16, int64_t E, int block,
                                         int bits, int N, int M, void* codes, float* scales,
                                         cudaStream_t s) {
  bool v8 = true;
  for (int t = 0; t < tab.count; ++t) v8 = v8 && (reinterpret_cast<uintptr_t>(tab.ptr[t]) & 31) == 0;
  return is_bf16 ? launch_reorder_quant_tensors_bf16(tab, E, block, bits, N, M, v8, codes, scales, s)
                 : launch_reorder_quant_tensors_f16(tab, E, block, bits, N, M, v8, codes, scales, s);
}

cudaError_t launch_reorder_quant(const void* grads, int is_bf16, int64_t E, int block, int bits,
                                 int N, int M, int l_begin, int l_end, int ranks, void* codes,
                                 float* scales, cudaStream_t s) {
  const bool v8 = (reinterpret_cast<uintptr_t>(grads) & 31) == 0;
  return by_type_bits_block(is_bf16, bits, block, v8, [&]<typename TT, int BITS, int B, bool V8>() {
    return run_reorder_quant<TT, BITS, B, V8>(grads, E, N, M, l_begin, l_end, ranks, codes,
                                              scales, s);
  });
}

}  // namespace zpp
