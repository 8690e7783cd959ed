// reorder_tensors.cuh -- K3T: the qgZ slice reorder + quantisation with the bucket flatten
// fused in (the bucket given as a list of tensors), instantiated per input type by
// reorder_tensors_f16.cu and reorder_tensors_bf16.cu so the two compile in parallel.
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
// (atlas.scime.ai summary), Approach: tensor-slice reordering for correct placement.
#pragma once

#include "quant_tile.cuh"

namespace zpp {

// K3 with the bucket flatten fused in: as k_reorder_quant (whole exchange), but every
// rank's bucket is read from its copies of the tensors in `tab` instead of a flat
// [W][E] buffer. The codes and scales are those of k_reorder_quant over the flattened
// bucket, bit for bit; the flattening copy (a full read and write of the bucket) is saved.
template <typename TT, int BITS, int B, bool V8>
__global__ void __launch_bounds__(kThreads)
    k_reorder_quant_tensors(const __grid_constant__ TensorTable tab, int64_t E, int N, int M,
                            uint8_t* __restrict__ codes, float* __restrict__ scales) {
  constexpr int TILE = QuantTile<B>::TILE;
  const int lane = threadIdx.x & 31;
  const int64_t k = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
  const int p = blockIdx.y, r = blockIdx.z;
  if (k * TILE < S) {
    const int l_d = p / N, n_d = p - l_d * N;
    const int64_t j = static_cast<int64_t>(n_d) * M + l_d;
    const int64_t base = j * S + k * TILE;
    const int64_t out_off = r * E + p * S + k * TILE;
    const int64_t rem = S - k * TILE;
    const TensorHit h = find_tensor(tab, base, lane);  // warp-uniform: k is per warp
    uint8_t* c = codes + out_off * BITS / 8;
    float* sc = scales + out_off / B;
    if (base + (rem < TILE ? rem : TILE) <= h.end) {  // the tile lies in one tensor
      const FlatSrc<V8> src{h.ptr + r * (h.end - h.start) + (base - h.start)};
      if (rem >= TILE) quant_tile<TT, BITS, B, true>(src, c, sc, TILE, lane);
      else quant_tile<TT, BITS, B, false>(src, c, sc, static_cast<int>(rem), lane);
    } else {
      const TensorSrc<V8> src{tab, base, r};
      if (rem >= TILE) quant_tile<TT, BITS, B, true>(src, c, sc, TILE, lane);
      else quant_tile<TT, BITS, B, false>(src, c, sc, static_cast<int>(rem), lane);
    }
  }
}

// K3T for one input type TT: dispatch over (bits, block, 256-bit loads).
template <typename TT>
cudaError_t run_reorder_quant_tensors(const TensorTable& tab, int64_t E, int block, int bits,
                                      int N, int M, bool v8, void* codes, float* scales,
                                      cudaStream_t s) {
  auto launch = [&]<typename T2, int BITS, int B, bool V8>() {
    const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
    const int64_t tps = (S + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
    const dim3 grid(tile_grid(tps, kWarps), static_cast<unsigned>(W), static_cast<unsigned>(W));
    k_reorder_quant_tensors<T2, BITS, B, V8><<<grid, kThreads, 0, s>>>(
        tab, E, N, M, static_cast<uint8_t*>(codes), scales);
    return cudaGetLastError();
  };
  return v8 ? by_bits_block<TT, true>(bits, block, launch)
            : by_bits_block<TT, false>(bits, block, launch);
}

}  // namespace zpp
