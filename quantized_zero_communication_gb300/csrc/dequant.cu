// dequant.cu -- K2: qwZ dequantisation after the all-gather, y = (float)q * scale rounded
// into fp16, bf16 or fp32.
//
// Warp tile (one per warp): 4 rows of 512 elements. Per row a lane reads 16 codes (16 bytes INT8, 8
// bytes INT4) and one block scale (the 16 elements never straddle a block, block >= 64)
// and writes 16 outputs with 256-bit stores (one for fp16/bf16, two for fp32), so a
// warp store instruction covers 1-2 KiB of contiguous output.
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
// (atlas.scime.ai summary), Approach; "ZeRO++: ... Giant Model Training" (mlsanity.com),
// Abstract: block-quantisation based all-gather.
#include <type_traits>

#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

constexpr int kDqVec = 16;                 // elements per lane per row
constexpr int kDqRow = 32 * kDqVec;        // 512
constexpr int kDqRows = 4;
constexpr int kDqTile = kDqRows * kDqRow;  // 2048 elements per warp tile

template <int BITS>
__device__ __forceinline__ void load_codes16(const uint8_t* p, uint32_t w[4]) {
  if constexpr (BITS == 8) {
    uint4 v = ld_stream_v4(p);
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  } else {
    uint2 v = ld_stream_v2(p);
    w[0] = v.x, w[1] = v.y, w[2] = 0u, w[3] = 0u;
  }
}

// 16 codes -> 16 dequantised fp32 values in element order, y = fl((float)q * s).
template <int BITS>
__device__ __forceinline__ void dequant16(const uint32_t w[4], float s, float v[16]) {
  const f32x2 ss = f2(s, s);
  if constexpr (BITS == 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f32x2 q[2];
      int8x4_to_f2(w[k], q);
      f2_split(f2_mul(q[0], ss), v[4 * k], v[4 * k + 1]);
      f2_split(f2_mul(q[1], ss), v[4 * k + 2], v[4 * k + 3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      f32x2 q[4];
      int4x8_to_f2(w[k], q);
#pragma unroll
      for (int j = 0; j < 4; ++j) f2_split(f2_mul(q[j], ss), v[8 * k + 2 * j], v[8 * k + 2 * j + 1]);
    }
  }
}

template <typename OT>
__device__ __forceinline__ void store1(void* y, int64_t e, float v) {
  if constexpr (std::is_same_v<OT, OutF32>)
    static_cast<float*>(y)[e] = v;
  else if constexpr (std::is_same_v<OT, OutF16>)
    static_cast<__half*>(y)[e] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(y)[e] = __float2bfloat16_rn(v);
}

template <int BITS, typename OT, bool V8>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t* __restrict__ codes,
                                                      const float* __restrict__ scales,
                                                      int64_t n, int log2b, void* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t full = n / kDqTile;
  if (t < full) {
    uint32_t w[kDqRows][4];
    float s[kDqRows];
#pragma unroll
    for (int u = 0; u < kDqRows; ++u) {
      const int64_t e = t * kDqTile + u * kDqRow + lane * kDqVec;
      load_codes16<BITS>(codes + e * BITS / 8, w[u]);
      s[u] = __ldg(scales + (e >> log2b));
    }
#pragma unroll
    for (int u = 0; u < kDqRows; ++u) {
      const int64_t e = t * kDqTile + u * kDqRow + lane * kDqVec;
      float v[kDqVec];
      dequant16<BITS>(w[u], s[u], v);
      store16<OT, V8>(y, e, v);
    }
  } else if (t == full) {
    // Ragged end: element-wise.
    for (int64_t e = full * kDqTile + lane; e < n; e += 32) {
      const int code = BITS == 8 ? static_cast<int>(static_cast<int8_t>(__ldg(codes + e)))
                                 : code_int4(__ldg(codes + (e >> 1)), static_cast<int>(e & 1));
      store1<OT>(y, e, __fmul_rn(static_cast<float>(code), __ldg(scales + (e >> log2b))));
    }
  }
}

template <int BITS, typename OT>
static cudaError_t run_dequant(const void* codes, const float* scales, int64_t n, int log2b,
                               void* y, cudaStream_t s) {
  const int64_t tiles = (n + kDqTile - 1) / kDqTile;
  const int grid = tile_grid(tiles, kWarps);
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  if ((reinterpret_cast<uintptr_t>(y) & 31) == 0)
    k_dequant<BITS, OT, true><<<grid, kThreads, 0, s>>>(c, scales, n, log2b, y);
  else
    k_dequant<BITS, OT, false><<<grid, kThreads, 0, s>>>(c, scales, n, log2b, y);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const void* codes, const float* scales, int64_t n, int block, int bits,
                           void* y, int out_kind, cudaStream_t s) {
  const int log2b = __builtin_ctz(static_cast<unsigned>(block));
  if (bits == 8) {
    if (out_kind == 0) return run_dequant<8, OutF16>(codes, scales, n, log2b, y, s);
    if (out_kind == 1) return run_dequant<8, OutBF16>(codes, scales, n, log2b, y, s);
    return run_dequant<8, OutF32>(codes, scales, n, log2b, y, s);
  }
  if (out_kind == 0) return run_dequant<4, OutF16>(codes, scales, n, log2b, y, s);
  if (out_kind == 1) return run_dequant<4, OutBF16>(codes, scales, n, log2b, y, s);
  return run_dequant<4, OutF32>(codes, scales, n, log2b, y, s);
}

}  // namespace zpp
