// quant.cu -- K1 (qwZ block quantisation) and K3 (qgZ slice reorder + quantisation).
//
// Both run the same warp tile: a warp owns TILE = max(block, 2048) consecutive
// elements, each lane loads 16 of them per row with one 256-bit load (a row is 512
// elements, 1 KiB of fp16/bf16), all rows of the tile are in flight before any
// arithmetic, the block absmax is taken on the sign-cleared 16-bit patterns (two per
// instruction) and reduced with warp shuffles, and each lane packs its 16 codes into
// one 16-byte (INT8) or 8-byte (INT4) store. Every input byte is read exactly once.
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model
// Training" (atlas.scime.ai summary), Approach: block-wise INT8 weight quantisation,
// INT4 gradients, tensor-slice reordering for correct placement. "LIT-102: ZeRO++ ..."
// Key takeaways: block-wise rather than per-tensor scales.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

// Where a warp tile's input elements come from. FlatSrc: one contiguous run that starts at
// the tile's first element. vec(off) loads the 16 elements at tile offset off (a multiple
// of 16) as one 256-bit vector; elem(off) loads one element.
struct FlatSrc {
  const uint16_t* p;
  __device__ __forceinline__ U8x32 vec(int off) const { return ld_stream_v8(p + off); }
  __device__ __forceinline__ uint16_t elem(int off) const { return __ldg(p + off); }
};

// The fused bucket flatten: rank r's bucket is the concatenation of its copies of the
// tensors in `tab`, so bucket element i is element i - offs[t] of rank r's copy of tensor
// t, where offs[t] <= i < offs[t+1]. Tensor t holds the W ranks' copies back to back, rank
// r's at ptr[t] + r * (offs[t+1] - offs[t]); tensors are multiples of 16 elements, so no
// 16-element vector straddles two of them.
struct TensorHit {
  const uint16_t* ptr;
  int64_t start, end;  // offs[t], offs[t+1]
};

// Warp-collective (all 32 lanes, converged): the tensor holding the warp-uniform bucket
// element a (0 <= a < E). Lanes test 32 candidate ends at once and a ballot counts those
// <= a (the ends are non-decreasing, so the true ones form a prefix): one round of table
// loads for up to 32 tensors, two (a coarse pass at stride ceil(T/32) first) for more.
__device__ __forceinline__ TensorHit find_tensor(const TensorTable& tab, int64_t a, int lane) {
  const int T = tab.count;
  int lo = 0;
  if (T > 32) {
    const int step = (T + 31) >> 5;
    lo = __popc(__ballot_sync(~0u, tab.offs[min((lane + 1) * step, T)] <= a)) * step;
  }
  const int64_t end = tab.offs[min(lo + lane + 1, T)];
  const int64_t start = tab.offs[min(lo + lane, T)];
  const uint16_t* p = tab.ptr[min(lo + lane, T - 1)];
  const int d = __popc(__ballot_sync(~0u, end <= a));  // tensor lo + d, held by lane d
  return TensorHit{reinterpret_cast<const uint16_t*>(__shfl_sync(
                       ~0u, reinterpret_cast<unsigned long long>(p), d)),
                   __shfl_sync(~0u, start, d), __shfl_sync(~0u, end, d)};
}

// Input of a warp tile of rank r's bucket that spans several tensors (a tile inside one
// tensor is read as a FlatSrc run): each load looks its tensor up by binary search.
struct TensorSrc {
  const TensorTable& tab;
  int64_t base;  // bucket index of the tile's first element
  int64_t r;     // source rank
  __device__ __forceinline__ const uint16_t* at(int64_t i) const {
    int lo = 0, hi = tab.count;  // invariant: offs[lo] <= i < offs[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tab.offs[mid] <= i) lo = mid;
      else hi = mid;
    }
    const int64_t len = tab.offs[lo + 1] - tab.offs[lo];
    return tab.ptr[lo] + r * len + (i - tab.offs[lo]);
  }
  __device__ __forceinline__ U8x32 vec(int off) const { return ld_stream_v8(at(base + off)); }
  __device__ __forceinline__ uint16_t elem(int off) const { return __ldg(at(base + off)); }
};

template <int B>
struct QuantTile {
  static constexpr int VEC = 16;                      // elements per lane per row
  static constexpr int ROW = 32 * VEC;                // 512 elements per warp row
  static constexpr int TILE = B > 2048 ? B : 2048;    // elements per warp tile
  static constexpr int ROWS = TILE / ROW;
};

// Quantise one warp tile. `in` gives the tile's input elements (FlatSrc or TensorSrc),
// `codes` points at its first code byte, `scales` at its first block scale. FULL: all TILE
// elements valid; otherwise only the first `valid` (any count; lanes past it load zeros,
// which leave the absmax unchanged and give code 0, and store nothing).
template <typename TT, int BITS, int B, bool FULL, typename Src>
__device__ __forceinline__ void quant_tile(const Src& in, uint8_t* __restrict__ codes,
                                           float* __restrict__ scales, int valid, int lane) {
  using T = QuantTile<B>;
  constexpr int VEC = T::VEC, ROW = T::ROW, ROWS = T::ROWS;
  U8x32 raw[ROWS];
  int cnt[ROWS];
#pragma unroll
  for (int u = 0; u < ROWS; ++u) {
    const int off = u * ROW + lane * VEC;
    if (FULL) {
      cnt[u] = VEC;
      raw[u] = in.vec(off);
    } else {
      int c = valid - off;
      c = c < 0 ? 0 : (c > VEC ? VEC : c);
      cnt[u] = c;
      if (c == VEC) {
        raw[u] = in.vec(off);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) raw[u].w[k] = 0u;
        for (int i = 0; i < c; ++i)
          raw[u].w[i >> 1] |= static_cast<uint32_t>(in.elem(off + i)) << (16 * (i & 1));
      }
    }
  }

  // Block absmax -> scale and inverse for every row.
  float sc[ROWS], iv[ROWS];
  if constexpr (B < ROW) {
    constexpr int LPB = B / VEC;  // lanes per block (4, 8 or 16)
#pragma unroll
    for (int u = 0; u < ROWS; ++u) {
      uint32_t a = warp_max_u32(absmax_bits16<8>(raw[u].w), LPB);
      block_scale<BITS>(bits16_to_float(a, TT()), sc[u], iv[u]);
    }
  } else {
    constexpr int RPB = B / ROW;  // rows per block
#pragma unroll
    for (int b = 0; b < ROWS / RPB; ++b) {
      uint32_t a = absmax_bits16<8>(raw[b * RPB].w);
#pragma unroll
      for (int i = 1; i < RPB; ++i) a = max(a, absmax_bits16<8>(raw[b * RPB + i].w));
      a = warp_max_u32(a, 32);
      float s, v;
      block_scale<BITS>(bits16_to_float(a, TT()), s, v);
#pragma unroll
      for (int i = 0; i < RPB; ++i) {
        sc[b * RPB + i] = s;
        iv[b * RPB + i] = v;
      }
    }
  }

  // Codes: 16 per lane per row, rounded with the magic-number addition (see round_codes).
#pragma unroll
  for (int u = 0; u < ROWS; ++u) {
    const int off = u * ROW + lane * VEC;
    const f32x2 iv2 = f2(iv[u], iv[u]);
    f32x2 r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 f = unpack2(raw[u].w[k], TT());
      r[k] = round_codes(f2(f.x, f.y), iv2);
    }
    if constexpr (BITS == 8) {
      const uint4 v = make_uint4(pack_int8x4(r), pack_int8x4(r + 2), pack_int8x4(r + 4),
                                 pack_int8x4(r + 6));
      if (FULL || cnt[u] == VEC) {
        st_v4(codes + off, v);
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        for (int i = 0; i < cnt[u]; ++i) codes[off + i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
      }
    } else {
      const uint2 v = make_uint2(pack_int4x8(r), pack_int4x8(r + 4));
      if (FULL || cnt[u] == VEC) {
        st_v2(codes + off / 2, v);
      } else {
        const uint32_t w[2] = {v.x, v.y};
        const int nbytes = (cnt[u] + 1) / 2;
        for (int i = 0; i < nbytes; ++i) codes[off / 2 + i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
      }
    }
  }

  // Scales: one lane per block.
  if constexpr (B < ROW) {
    constexpr int LPB = B / VEC;
#pragma unroll
    for (int u = 0; u < ROWS; ++u) {
      const int e0 = u * ROW + lane * VEC;
      if ((lane % LPB) == 0 && (FULL || e0 < valid)) scales[e0 / B] = sc[u];
    }
  } else {
    constexpr int RPB = B / ROW;
#pragma unroll
    for (int b = 0; b < ROWS / RPB; ++b)
      if (lane == 0 && (FULL || b * B < valid)) scales[b] = sc[b * RPB];
  }
}

// K1: x[n] -> codes, scales. One warp tile per warp (a grid of one tile per warp streams
// HBM better on this part than a persistent grid-stride loop); the warp that owns the
// ragged last tile takes the bounds-checked path.
template <typename TT, int BITS, int B>
__global__ void __launch_bounds__(kThreads) k_quant(const uint16_t* __restrict__ x, int64_t n,
                                                    uint8_t* __restrict__ codes,
                                                    float* __restrict__ scales) {
  constexpr int TILE = QuantTile<B>::TILE;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t full = n / TILE;
  if (t < full) {
    quant_tile<TT, BITS, B, true>(FlatSrc{x + t * TILE}, codes + t * (TILE * BITS / 8),
                                  scales + t * (TILE / B), TILE, lane);
  } else if (t == full && n > full * TILE) {
    quant_tile<TT, BITS, B, false>(FlatSrc{x + t * TILE}, codes + t * (TILE * BITS / 8),
                                   scales + t * (TILE / B), static_cast<int>(n - t * TILE), lane);
  }
}

// K3: per source rank r, output slice position p = l_d*N + n_d holds original slice
// j = n_d*M + l_d. Grid (tile group, p - p_begin, r): each warp owns one warp tile of
// slice p of rank r (the last tile of a slice may be short but always holds whole
// blocks). A launch may cover only the slices of some hop-1 chunks (p_begin = l_begin*N).
template <typename TT, int BITS, int B>
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
      quant_tile<TT, BITS, B, true>(FlatSrc{grads + in_off}, codes + out_off * BITS / 8,
                                    scales + out_off / B, TILE, lane);
    else
      quant_tile<TT, BITS, B, false>(FlatSrc{grads + in_off}, codes + out_off * BITS / 8,
                                     scales + out_off / B, static_cast<int>(rem), lane);
  }
}

// K3 with the bucket flatten fused in: as k_reorder_quant (whole exchange), but every
// rank's bucket is read from its copies of the tensors in `tab` instead of a flat
// [W][E] buffer. The codes and scales are those of k_reorder_quant over the flattened
// bucket, bit for bit; the flattening copy (a full read and write of the bucket) is saved.
template <typename TT, int BITS, int B>
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
      const FlatSrc src{h.ptr + r * (h.end - h.start) + (base - h.start)};
      if (rem >= TILE) quant_tile<TT, BITS, B, true>(src, c, sc, TILE, lane);
      else quant_tile<TT, BITS, B, false>(src, c, sc, static_cast<int>(rem), lane);
    } else {
      const TensorSrc src{tab, base, r};
      if (rem >= TILE) quant_tile<TT, BITS, B, true>(src, c, sc, TILE, lane);
      else quant_tile<TT, BITS, B, false>(src, c, sc, static_cast<int>(rem), lane);
    }
  }
}

template <typename TT, int BITS, int B>
static cudaError_t run_quant(const void* x, int64_t n, void* codes, float* scales, cudaStream_t s) {
  auto kern = k_quant<TT, BITS, B>;
  const int64_t tiles = (n + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
  const int grid = tile_grid(tiles, kWarps);
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), n, static_cast<uint8_t*>(codes),
                                 scales);
  return cudaGetLastError();
}

template <typename TT, int BITS, int B>
static cudaError_t run_reorder_quant(const void* g, int64_t E, int N, int M, int l_begin, int l_end,
                                     void* codes, float* scales, cudaStream_t s) {
  auto kern = k_reorder_quant<TT, BITS, B>;
  const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
  const int64_t tps = (S + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
  // output slice positions of chunks l_begin .. l_end-1: p in [l_begin*N, l_end*N)
  const dim3 grid(tile_grid(tps, kWarps), static_cast<unsigned>((l_end - l_begin) * N),
                  static_cast<unsigned>(W));
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(g), E, N, M, l_begin * N,
                                 static_cast<uint8_t*>(codes), scales);
  return cudaGetLastError();
}

// Compile-time dispatch over (dtype, bits, block).
template <typename TT, int BITS, typename F>
static cudaError_t by_block(int block, F&& f) {
  switch (block) {
    case 64: return f.template operator()<TT, BITS, 64>();
    case 128: return f.template operator()<TT, BITS, 128>();
    case 256: return f.template operator()<TT, BITS, 256>();
    case 512: return f.template operator()<TT, BITS, 512>();
    case 1024: return f.template operator()<TT, BITS, 1024>();
    case 2048: return f.template operator()<TT, BITS, 2048>();
    case 4096: return f.template operator()<TT, BITS, 4096>();
    default: return cudaErrorInvalidValue;
  }
}

template <typename F>
static cudaError_t by_type_bits_block(int is_bf16, int bits, int block, F&& f) {
  if (is_bf16)
    return bits == 8 ? by_block<BF16, 8>(block, f) : by_block<BF16, 4>(block, f);
  return bits == 8 ? by_block<F16, 8>(block, f) : by_block<F16, 4>(block, f);
}

cudaError_t launch_quant(const void* x, int is_bf16, int64_t n, int block, int bits, void* codes,
                         float* scales, cudaStream_t s) {
  return by_type_bits_block(is_bf16, bits, block, [&]<typename TT, int BITS, int B>() {
    return run_quant<TT, BITS, B>(x, n, codes, scales, s);
  });
}

cudaError_t launch_reorder_quant_tensors(const TensorTable& tab, int is_bf16, int64_t E, int block,
                                         int bits, int N, int M, void* codes, float* scales,
                                         cudaStream_t s) {
  return by_type_bits_block(is_bf16, bits, block, [&]<typename TT, int BITS, int B>() {
    const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
    const int64_t tps = (S + QuantTile<B>::TILE - 1) / QuantTile<B>::TILE;
    const dim3 grid(tile_grid(tps, kWarps), static_cast<unsigned>(W), static_cast<unsigned>(W));
    k_reorder_quant_tensors<TT, BITS, B><<<grid, kThreads, 0, s>>>(
        tab, E, N, M, static_cast<uint8_t*>(codes), scales);
    return cudaGetLastError();
  });
}

cudaError_t launch_reorder_quant(const void* grads, int is_bf16, int64_t E, int block, int bits,
                                 int N, int M, int l_begin, int l_end, void* codes, float* scales,
                                 cudaStream_t s) {
  return by_type_bits_block(is_bf16, bits, block, [&]<typename TT, int BITS, int B>() {
    return run_reorder_quant<TT, BITS, B>(grads, E, N, M, l_begin, l_end, codes, scales, s);
  });
}

}  // namespace zpp
