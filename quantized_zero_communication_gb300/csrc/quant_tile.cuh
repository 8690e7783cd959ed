// quant_tile.cuh -- the warp tile shared by K1 (qwZ block quantisation) and K3 / K3T
// (qgZ slice reorder + quantisation), its input sources, and the launch-time dispatch.
//
// A warp owns TILE = max(block, 2048) consecutive elements, each lane loads 16 of them
// per row with one 256-bit load (two 128-bit loads when the input is only 16-byte
// aligned; a row is 512 elements, 1 KiB of fp16/bf16), all rows of the tile are in flight
// before any arithmetic, the block absmax is taken on the sign-cleared 16-bit patterns
// (two per instruction) and reduced with warp shuffles, and each lane packs its 16 codes
// into one 16-byte (INT8) or 8-byte (INT4) store. Every input byte is read exactly once.
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model
// Training" (atlas.scime.ai summary), Approach: block-wise INT8 weight quantisation,
// INT4 gradients, tensor-slice reordering for correct placement. "LIT-102: ZeRO++ ..."
// Key takeaways: block-wise rather than per-tensor scales.
#pragma once

#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

// Where a warp tile's input elements come from. FlatSrc: one contiguous run that starts at
// the tile's first element. vec(off) loads the 16 elements at tile offset off (a multiple
// of 16) as one 256-bit vector; elem(off) loads one element.
// V8: the run starts 32-byte aligned (one 256-bit load per vector); otherwise it starts
// 16-byte aligned and each vector is two 128-bit loads.
template <bool V8>
struct FlatSrc {
  const uint16_t* p;
  __device__ __forceinline__ U8x32 vec(int off) const { return ld_vec32<V8>(p + off); }
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
template <bool V8>
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
  __device__ __forceinline__ U8x32 vec(int off) const { return ld_vec32<V8>(at(base + off)); }
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

// Compile-time dispatch over (dtype, bits, block, 256-bit input vectors).
template <typename TT, int BITS, bool V8, typename F>
static cudaError_t by_block(int block, F&& f) {
  switch (block) {
    case 64: return f.template operator()<TT, BITS, 64, V8>();
    case 128: return f.template operator()<TT, BITS, 128, V8>();
    case 256: return f.template operator()<TT, BITS, 256, V8>();
    case 512: return f.template operator()<TT, BITS, 512, V8>();
    case 1024: return f.template operator()<TT, BITS, 1024, V8>();
    case 2048: return f.template operator()<TT, BITS, 2048, V8>();
    case 4096: return f.template operator()<TT, BITS, 4096, V8>();
    default: return cudaErrorInvalidValue;
  }
}

template <typename TT, bool V8, typename F>
static cudaError_t by_bits_block(int bits, int block, F&& f) {
  return bits == 8 ? by_block<TT, 8, V8>(block, f) : by_block<TT, 4, V8>(block, f);
}

template <typename F>
static cudaError_t by_type_bits_block(int is_bf16, int bits, int block, bool v8, F&& f) {
  if (is_bf16)
    return v8 ? by_bits_block<BF16, true>(bits, block, f) : by_bits_block<BF16, false>(bits, block, f);
  return v8 ? by_bits_block<F16, true>(bits, block, f) : by_bits_block<F16, false>(bits, block, f);
}

}  // namespace zpp
