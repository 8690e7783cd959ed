// quant.cu -- K1: qwZ block quantisation of a weight shard (INT8, also INT4), one warp
// tile per warp (see quant_tile.cuh).
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model
// Training" (atlas.scime.ai summary), Approach: block-wise INT8 weight quantisation.
// "LIT-102: ZeRO++ ..." Key takeaways: block-wise rather than per-tensor scales.
#include "quant_tile.cuh"

namespace zpp {

// K1: x[n] -> codes, scales. One warp tile per warp (a grid of one tile per warp streams
// HBM better on this part than a persistent grid-stride loop); the warp that owns the
// ragged last tile takes the bounds-checked path.
template <typename TT, int BITS, int B, bool V8>
__global__ void __launch_bounds__(kThreads) k_quant(const uint16_t* __restrict__ x, int64_t n,
                                                    uint8_t* __restrict__ codes,
                                                    float* __restrict__ scales) {
  constexpr int TILE = QuantTile<B>::TILE;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t full = n / TILE;
  if (t < full) {
    quant_tile<TT, BITS, B, true>(FlatSrc<V8>{x + t * TILE}, codes + t * (TILE * BITS / 8),
                                  scales + t * (TILE / B), TILE, lane);
  } else if (t == full && n > full * TILE) {
    quant_tile<TT, BITS, B, false>(FlatSrc<V8>{x + t * TILE}, codes + t * (TILE * BITS / 8),
                                   scales + t * (TILE / B), static_cast<int>(n - t * TILE), lane);
  }
}

template <typename TT, int BITS, int B, bool V8>
static cudaError_t run_quant(const void* x, int64_t n, void* codes, float* scales, cudaStream_t s) {
  auto kern = k_quant<TT, BITS, B, V8>;
  const int64_t tiles = (n + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
  const int grid = tile_grid(tiles, kWarps);
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), n, static_cast<uint8_t*>(codes),
                                 scales);
  return cudaGetLastError();
}

cudaError_t launch_quant(const void* x, int is_bf16, int64_t n, int block, int bits, void* codes,
                         float* scales, cudaStream_t s) {
  const bool v8 = (reinterpret_cast<uintptr_t>(x) & 31) == 0;
  return by_type_bits_block(is_bf16, bits, block, v8, [&]<typename TT, int BITS, int B, bool V8>() {
    return run_quant<TT, BITS, B, V8>(x, n, codes, scales, s);
  });
}

}  // namespace zpp
