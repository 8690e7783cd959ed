// qgz.cu -- the two reduction hops of qgZ on virtual ranks laid out in HBM.
//
// K4 (intra-node hop, the pages' fusion kernel): receiver (n, l) reads chunk l of the M
// ranks of node n straight from their reordered, quantised buffers (the all-to-all is
// an index map), dequantises, sums in fp32 in ascending source order, then requantises
// the sums by blocks -- one pass, every source code read once, sums kept in registers.
// K5 (inter-node hop): receiver (n, l) reads slice n of the hop-1 output of ranks
// (n', l), n' = 0..N-1, dequantises and sums into its fp32 owner slice.
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
// (atlas.scime.ai summary), Approach: 2-hop all-to-all INT4 gradient reduction that
// dequantises before reducing; Measured effects table: the fusion kernel.
// "LIT-102: ZeRO++ ..." Key takeaways: quantised once per exchange, reduced locally in
// higher precision.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

// acc (pairs of fp32 sums) += dequantised 16 code bytes with scale s: each term q * s is
// added with one rounding (fused multiply-add), in the order the sources are visited.
template <int BITS>
__device__ __forceinline__ void accumulate16B(f32x2* acc, const uint4& v, float s) {
  const f32x2 ss = f2(s, s);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (BITS == 8) {
      f32x2 q[2];
      int8x4_to_f2(w[k], q);
      acc[2 * k] = f2_fma(q[0], ss, acc[2 * k]);
      acc[2 * k + 1] = f2_fma(q[1], ss, acc[2 * k + 1]);
    } else {
      f32x2 q[4];
      int4x8_to_f2(w[k], q);
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[4 * k + j] = f2_fma(q[j], ss, acc[4 * k + j]);
    }
  }
}

// acc += dequantised 8 code bytes (INT4: 16 codes) or 16 code bytes (INT8: 16 codes).
template <int BITS>
__device__ __forceinline__ void accumulate16codes(f32x2* acc, const uint4& v, float s) {
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

// K4. CTA tile: 8 warps x one row each; a row is 32 lanes x EPL elements (one 16-byte
// code vector per lane and source). Blocks wider than a row are reduced across the
// warps that share them through shared memory.
template <int BITS, int KC>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce_requant(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                             int64_t E, int log2b, int N, int M, uint8_t* __restrict__ out_codes,
                             float* __restrict__ out_scales) {
  constexpr int EPL = BITS == 4 ? 32 : 16;
  constexpr int ROWLEN = 32 * EPL;
  constexpr int CT = kWarps * ROWLEN;
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = 1 << log2b;
  const int64_t W = static_cast<int64_t>(N) * M;
  const int64_t C = E / M;  // = N * S, the hop-1 chunk
  const int64_t tpr = (C + CT - 1) / CT;
  const int64_t total = W * tpr;
  const int64_t cb_in = E * BITS / 8, sc_in = E >> log2b;
  const int64_t cb_out = C * BITS / 8, sc_out = C >> log2b;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int64_t r = t / tpr, kk = t - r * tpr;
    const int n = static_cast<int>(r / M), l = static_cast<int>(r - static_cast<int64_t>(n) * M);
    const int64_t e = kk * CT + warp * ROWLEN + lane * EPL;
    const bool valid = e < C;
    const int64_t idx = static_cast<int64_t>(l) * C + e;  // chunk l of each source
    const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx * BITS / 8;
    const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);
    constexpr int NP = EPL / 2;  // fp32 pairs per lane
    f32x2 acc[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) acc[j] = f2(0.0f, 0.0f);
    for (int k0 = 0; k0 < M; k0 += KC) {
      uint4 raw[KC];
      float s[KC];
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        if (valid && k0 + i < M) {
          raw[i] = ld_stream_v4(cbase + (k0 + i) * cb_in);
          s[i] = __ldg(sbase + (k0 + i) * sc_in);
        } else {
          raw[i] = make_uint4(0u, 0u, 0u, 0u);
          s[i] = 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        if (k0 + i < M) accumulate16B<BITS>(acc, raw[i], s[i]);
      }
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      float a, b;
      f2_split(acc[j], a, b);
      m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
    }
    if (B <= ROWLEN) {
      m = warp_max(m, B / EPL);
    } else {
      m = warp_max(m, 32);
      if (lane == 0) red[warp] = m;
      __syncthreads();
      const int wpb = B / ROWLEN, w0 = warp & ~(wpb - 1);
      m = red[w0];
      for (int i = 1; i < wpb; ++i) m = fmaxf(m, red[w0 + i]);
      __syncthreads();
    }
    float sc, iv;
    block_scale<BITS>(m, sc, iv);
    if (valid) {
      const f32x2 iv2 = f2(iv, iv);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (BITS == 8) {
          const f32x2 r[2] = {round_codes(acc[2 * k], iv2), round_codes(acc[2 * k + 1], iv2)};
          w[k] = pack_int8x4(r);
        } else {
          const f32x2 r[4] = {round_codes(acc[4 * k], iv2), round_codes(acc[4 * k + 1], iv2),
                              round_codes(acc[4 * k + 2], iv2), round_codes(acc[4 * k + 3], iv2)};
          w[k] = pack_int4x8(r);
        }
      }
      const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
      st_v4(out_codes + r * cb_out + e * BITS / 8, v);
      if ((e & (B - 1)) == 0) out_scales[r * sc_out + (e >> log2b)] = sc;
    }
  }
}

// K5. A lane owns 16 consecutive outputs of its receiver's slice and writes them as two
// 256-bit stores (each a full 32-byte sector).
template <int BITS, int KC>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce(const uint8_t* __restrict__ codes, const float* __restrict__ scales, int64_t E,
                     int log2b, int N, int M, float* __restrict__ out) {
  constexpr int EPL = 16;
  constexpr int CT = kWarps * 32 * EPL;  // 4096 elements per CTA tile
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t W = static_cast<int64_t>(N) * M;
  const int64_t S = E / W, C = E / M;
  const int64_t tps = (S + CT - 1) / CT;
  const int64_t total = W * tps;
  const int64_t cb = C * BITS / 8, sc = C >> log2b;  // per hop-1 rank
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int64_t r = t / tps, kk = t - r * tps;
    const int n = static_cast<int>(r / M), l = static_cast<int>(r - static_cast<int64_t>(n) * M);
    const int64_t e = kk * CT + (warp * 32 + lane) * EPL;
    if (e >= S) continue;  // no barrier in this kernel
    const int64_t idx = static_cast<int64_t>(n) * S + e;  // slice n of each hop-1 output
    const uint8_t* cbase = codes + static_cast<int64_t>(l) * cb + idx * BITS / 8;
    const float* sbase = scales + static_cast<int64_t>(l) * sc + (idx >> log2b);
    const int64_t cstep = static_cast<int64_t>(M) * cb, sstep = static_cast<int64_t>(M) * sc;
    f32x2 acc[EPL / 2];
#pragma unroll
    for (int j = 0; j < EPL / 2; ++j) acc[j] = f2(0.0f, 0.0f);
    for (int k0 = 0; k0 < N; k0 += KC) {
      uint4 raw[KC];
      float s[KC];
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        if (k0 + i < N) {
          if constexpr (BITS == 8) {
            raw[i] = ld_stream_v4(cbase + (k0 + i) * cstep);
          } else {
            uint2 h = ld_stream_v2(cbase + (k0 + i) * cstep);
            raw[i] = make_uint4(h.x, h.y, 0u, 0u);
          }
          s[i] = __ldg(sbase + (k0 + i) * sstep);
        } else {
          raw[i] = make_uint4(0u, 0u, 0u, 0u);
          s[i] = 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        if (k0 + i < N) accumulate16codes<BITS>(acc, raw[i], s[i]);
      }
    }
    U8x32 a, b;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float lo, hi;
      f2_split(acc[j], lo, hi);
      a.w[2 * j] = __float_as_uint(lo);
      a.w[2 * j + 1] = __float_as_uint(hi);
      f2_split(acc[4 + j], lo, hi);
      b.w[2 * j] = __float_as_uint(lo);
      b.w[2 * j + 1] = __float_as_uint(hi);
    }
    float* p = out + r * S + e;
    st_v8(p, a);
    st_v8(p + 8, b);
  }
}

static int chunk_for(int k) { return k >= 8 ? 8 : (k > 2 ? 4 : (k == 2 ? 2 : 1)); }

template <int BITS, int KC>
static cudaError_t run_drr(const void* codes, const float* scales, int64_t E, int log2b, int N,
                           int M, void* out_codes, float* out_scales, cudaStream_t s) {
  auto kern = k_dequant_reduce_requant<BITS, KC>;
  static const int occ = occupancy_of(kern, kThreads);
  constexpr int CT = kWarps * 32 * (BITS == 4 ? 32 : 16);
  const int64_t C = E / M, W = static_cast<int64_t>(N) * M;
  const int grid = persistent_grid(W * ((C + CT - 1) / CT), occ);
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(codes), scales, E, log2b, N, M,
                                 static_cast<uint8_t*>(out_codes), out_scales);
  return cudaGetLastError();
}

template <int BITS, int KC>
static cudaError_t run_dr(const void* codes, const float* scales, int64_t E, int log2b, int N,
                          int M, float* out, cudaStream_t s) {
  auto kern = k_dequant_reduce<BITS, KC>;
  static const int occ = occupancy_of(kern, kThreads);
  constexpr int CT = kWarps * 32 * 16;
  const int64_t W = static_cast<int64_t>(N) * M, S = E / W;
  const int grid = persistent_grid(W * ((S + CT - 1) / CT), occ);
  kern<<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(codes), scales, E, log2b, N, M, out);
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
