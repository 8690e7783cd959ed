// qgz.cu -- the two reduction hops of qgZ on virtual ranks laid out in HBM.
//
// K4 (intra-node hop, the pages' fusion kernel): receiver (n, l) reads chunk l of the M
// ranks of node n straight from their reordered, quantised buffers (the all-to-all is
// an index map), dequantises, sums in fp32 in ascending source order, then requantises
// the sums by blocks -- one pass, every source code read once, sums kept in registers.
// K5 (inter-node hop): receiver (n, l) reads slice n of the hop-1 output of ranks
// (n', l), n' = 0..N-1, dequantises and sums into its fp32 owner slice.
//
// A lane owns 16 consecutive elements of its receiver (8 code bytes per source for INT4,
// 16 for INT8); its sums live in registers as eight fp32 pairs (2j, 2j+1).
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
// (atlas.scime.ai summary), Approach: 2-hop all-to-all INT4 gradient reduction that
// dequantises before reducing; Measured effects table: the fusion kernel.
// "LIT-102: ZeRO++ ..." Key takeaways: quantised once per exchange, reduced locally in
// higher precision.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

constexpr int kEpl = 16;               // elements per lane
constexpr int kRow = 32 * kEpl;        // 512 elements per warp row
constexpr int kCta = kWarps * kRow;    // 4096 elements per CTA tile

// 16 codes of one lane (INT4: words x, y; INT8: x, y, z, w).
template <int BITS>
__device__ __forceinline__ uint4 load_codes(const uint8_t* p) {
  if constexpr (BITS == 8) {
    return ld_stream_v4(p);
  } else {
    const uint2 h = ld_stream_v2(p);
    return make_uint4(h.x, h.y, 0u, 0u);
  }
}

// acc (eight fp32 pairs) += q * s for the lane's 16 codes: each term added with one
// rounding (fused multiply-add), in the order the sources are visited.
template <int BITS>
__device__ __forceinline__ void accumulate(f32x2 acc[8], const uint4& v, float s) {
  const f32x2 ss = f2(s, s);
  if constexpr (BITS == 8) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f32x2 q[2];
      int8x4_to_f2(w[k], q);
      acc[2 * k] = f2_fma(q[0], ss, acc[2 * k]);
      acc[2 * k + 1] = f2_fma(q[1], ss, acc[2 * k + 1]);
    }
  } else {
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      f32x2 q[4];
      int4x8_to_f2(w[k], q);
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[4 * k + j] = f2_fma(q[j], ss, acc[4 * k + j]);
    }
  }
}

// The lane's 16 values in element order.
__device__ __forceinline__ void unpair(const f32x2 acc[8], float out[16]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) f2_split(acc[j], out[2 * j], out[2 * j + 1]);
}

// K4. Grid (tile, l, n): CTA (x, l, n) owns tile x of receiver (n, l) -- 8 warps x one
// 512-element row each -- so no thread divides to find its work. Blocks wider than a row
// are reduced across the warps that share them through shared memory.
template <int BITS, int KC>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce_requant(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                             int64_t E, int log2b, int N, int M, uint8_t* __restrict__ out_codes,
                             float* __restrict__ out_scales) {
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = 1 << log2b;
  const int l = blockIdx.y, n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t C = E / M;  // = N * S, the hop-1 chunk
  const int64_t cb_in = E * BITS / 8, sc_in = E >> log2b;
  const int64_t cb_out = C * BITS / 8, sc_out = C >> log2b;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kCta + warp * kRow + lane * kEpl;
  const bool valid = e < C;  // C is a multiple of the block: whole blocks are in or out
  const int64_t idx = static_cast<int64_t>(l) * C + e;  // chunk l of each source
  const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);

  f32x2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = f2(0.0f, 0.0f);
  for (int k0 = 0; k0 < M; k0 += KC) {
    uint4 raw[KC];
    float s[KC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      if (valid && k0 + i < M) {
        raw[i] = load_codes<BITS>(cbase + (k0 + i) * cb_in);
        s[i] = __ldg(sbase + (k0 + i) * sc_in);
      } else {
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
        s[i] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < KC; ++i)
      if (k0 + i < M) accumulate<BITS>(acc, raw[i], s[i]);
  }

  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a, b;
    f2_split(acc[j], a, b);
    m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
  }
  if (B <= kRow) {
    m = warp_max(m, B / kEpl);
  } else {
    m = warp_max(m, 32);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    const int wpb = B / kRow, w0 = warp & ~(wpb - 1);
    m = red[w0];
    for (int i = 1; i < wpb; ++i) m = fmaxf(m, red[w0 + i]);
  }
  float sc, iv;
  block_scale<BITS>(m, sc, iv);
  if (!valid) return;
  const f32x2 iv2 = f2(iv, iv);
  uint8_t* dst = out_codes + r * cb_out + e * BITS / 8;
  if constexpr (BITS == 8) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const f32x2 q[2] = {round_codes(acc[2 * k], iv2), round_codes(acc[2 * k + 1], iv2)};
      w[k] = pack_int8x4(q);
    }
    st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
  } else {
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const f32x2 q[4] = {round_codes(acc[4 * k], iv2), round_codes(acc[4 * k + 1], iv2),
                          round_codes(acc[4 * k + 2], iv2), round_codes(acc[4 * k + 3], iv2)};
      w[k] = pack_int4x8(q);
    }
    st_v2(dst, make_uint2(w[0], w[1]));
  }
  if ((e & (B - 1)) == 0) out_scales[r * sc_out + (e >> log2b)] = sc;
}

// K5. Grid (tile, l, n) as for K4. A lane owns 16 consecutive outputs of its receiver's
// slice and writes them as two 256-bit stores (each a full 32-byte sector).
template <int BITS, int KC>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce(const uint8_t* __restrict__ codes, const float* __restrict__ scales, int64_t E,
                     int log2b, int N, int M, float* __restrict__ out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = blockIdx.y, n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t W = static_cast<int64_t>(N) * M;
  const int64_t S = E / W, C = E / M;
  const int64_t cb = C * BITS / 8, sc = C >> log2b;  // per hop-1 rank
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kCta + warp * kRow + lane * kEpl;
  if (e >= S) return;  // no barrier in this kernel
  const int64_t idx = static_cast<int64_t>(n) * S + e;  // slice n of each hop-1 output
  const uint8_t* cbase = codes + static_cast<int64_t>(l) * cb + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(l) * sc + (idx >> log2b);
  const int64_t cstep = static_cast<int64_t>(M) * cb, sstep = static_cast<int64_t>(M) * sc;

  f32x2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = f2(0.0f, 0.0f);
  for (int k0 = 0; k0 < N; k0 += KC) {
    uint4 raw[KC];
    float s[KC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      if (k0 + i < N) {
        raw[i] = load_codes<BITS>(cbase + (k0 + i) * cstep);
        s[i] = __ldg(sbase + (k0 + i) * sstep);
      } else {
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
        s[i] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < KC; ++i)
      if (k0 + i < N) accumulate<BITS>(acc, raw[i], s[i]);
  }
  float v[16];
  unpair(acc, v);
  U8x32 a, b;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a.w[j] = __float_as_uint(v[j]);
    b.w[j] = __float_as_uint(v[8 + j]);
  }
  float* p = out + r * S + e;
  st_v8(p, a);
  st_v8(p + 8, b);
}

static int chunk_for(int k) { return k >= 8 ? 8 : (k > 2 ? 4 : (k == 2 ? 2 : 1)); }

template <int BITS, int KC>
static cudaError_t run_drr(const void* codes, const float* scales, int64_t E, int log2b, int N,
                           int M, void* out_codes, float* out_scales, cudaStream_t s) {
  const int64_t C = E / M;
  const dim3 grid(tile_grid(C, kCta), M, N);
  k_dequant_reduce_requant<BITS, KC><<<grid, kThreads, 0, s>>>(
      static_cast<const uint8_t*>(codes), scales, E, log2b, N, M, static_cast<uint8_t*>(out_codes),
      out_scales);
  return cudaGetLastError();
}

template <int BITS, int KC>
static cudaError_t run_dr(const void* codes, const float* scales, int64_t E, int log2b, int N,
                          int M, float* out, cudaStream_t s) {
  const int64_t S = E / (static_cast<int64_t>(N) * M);
  const dim3 grid(tile_grid(S, kCta), M, N);
  k_dequant_reduce<BITS, KC><<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(codes), scales,
                                                       E, log2b, N, M, out);
  return cudaGetLastError();
}

template <int BITS>
static cudaError_t drr_bits(const void* c, const float* sc, int64_t E, int log2b, int N, int M,
                            void* oc, float* os, cudaStream_t s) {
  switch (chunk_for(M)) {
    case 8: return run_drr<BITS, 8>(c, sc, E, log2b, N, M, oc, os, s);
    case 4: return run_drr<BITS, 4>(c, sc, E, log2b, N, M, oc, os, s);
    case 2: return run_drr<BITS, 2>(c, sc, E, log2b, N, M, oc, os, s);
    default: return run_drr<BITS, 1>(c, sc, E, log2b, N, M, oc, os, s);
  }
}

template <int BITS>
static cudaError_t dr_bits(const void* c, const float* sc, int64_t E, int log2b, int N, int M,
                           float* out, cudaStream_t s) {
  switch (chunk_for(N)) {
    case 8: return run_dr<BITS, 8>(c, sc, E, log2b, N, M, out, s);
    case 4: return run_dr<BITS, 4>(c, sc, E, log2b, N, M, out, s);
    case 2: return run_dr<BITS, 2>(c, sc, E, log2b, N, M, out, s);
    default: return run_dr<BITS, 1>(c, sc, E, log2b, N, M, out, s);
  }
}

cudaError_t launch_dequant_reduce_requant(const void* codes, const float* scales, int64_t E,
                                          int block, int bits, int N, int M, void* out_codes,
                                          float* out_scales, cudaStream_t s) {
  const int log2b = __builtin_ctz(static_cast<unsigned>(block));
  return bits == 8 ? drr_bits<8>(codes, scales, E, log2b, N, M, out_codes, out_scales, s)
                   : drr_bits<4>(codes, scales, E, log2b, N, M, out_codes, out_scales, s);
}

cudaError_t launch_dequant_reduce(const void* codes, const float* scales, int64_t E, int block,
                                  int bits, int N, int M, float* out, cudaStream_t s) {
  const int log2b = __builtin_ctz(static_cast<unsigned>(block));
  return bits == 8 ? dr_bits<8>(codes, scales, E, log2b, N, M, out, s)
                   : dr_bits<4>(codes, scales, E, log2b, N, M, out, s);
}

}  // namespace zpp
