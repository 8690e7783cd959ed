// qgz.cu -- the two reduction hops of qgZ on virtual ranks laid out in HBM.
//
// K4 (intra-node hop, the pages' fusion kernel): receiver (n, l) reads chunk l of the M
// ranks of node n straight from their reordered, quantised buffers (the all-to-all is
// an index map), dequantises, sums in fp32 in ascending source order, then requantises
// the sums by blocks -- one pass, every source code read once, sums kept in registers.
// K5 (inter-node hop): receiver (n, l) reads slice n of the hop-1 output of ranks
// (n', l), n' = 0..N-1, dequantises and sums into its fp32 owner slice.
//
// A K4 lane reads 16 code bytes per source (32 INT4 or 16 INT8 elements); a K5 lane owns
// 16 elements. Sums live in registers as fp32 pairs, four pairs per code word k: elements
// (8k+2j, 8k+2j+1) -- except the INT4 words that K4 converts by the split integer / fp32
// path (k < kSplitWords), whose pairs hold (8k, 8k+2), (8k+4, 8k+6), (8k+1, 8k+3),
// (8k+5, 8k+7).
//
// Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
// (atlas.scime.ai summary), Approach: 2-hop all-to-all INT4 gradient reduction that
// dequantises before reducing; Measured effects table: the fusion kernel.
// "LIT-102: ZeRO++ ..." Key takeaways: quantised once per exchange, reduced locally in
// higher precision.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

// Lanes own 16 code bytes per source in K4 (32 INT4 / 16 INT8 elements; 32 INT8 codes in
// the wide kernel) and 16 elements in K5; a CTA tile is 8 warps x one row (4 warps in the
// INT4 staged, the prefetching and the wide kernels).
//
// K4 kernels, chosen per launch by drr_bits / run_drr (all give the same bits):
//   k_dequant_reduce_requant_ring8<KC>          INT8 codes, M >= 3: the bulk-copy ring below;
//   k_dequant_reduce_requant_wide8<KC, V8>      INT8 codes, M = 1 or 2: the full tiles, 32
//       outputs per lane, the codes loaded straight into registers;
//   k_dequant_reduce_requant_prefetch<KC>       INT4 codes, M = 1 or 2: the full tiles, two
//       per CTA, both loaded into registers before the first is converted;
//   k_dequant_reduce_requant_staged<BITS, KC, SPLIT>  INT4 with M = KC in {4, 8} or
//       M = 16: the full tiles, the sources' codes staged in shared memory by cp.async;
//   k_dequant_reduce_requant_split<KC>          INT4, M a multiple of a 4- or 8-source
//       chunk otherwise, and the ragged last tile of a staged launch;
//   k_dequant_reduce_requant<BITS, KC, EXACT>   otherwise: INT4 with M not a multiple of
//       its chunk, and the ragged last tile of a prefetching or a wide launch.
// With chunks of 4 or more sources, kSplitWords of the 4 code words per source go through
// int4x8_to_f2_eo, which shares the conversion between the integer and fp32 pipes. Measured
// on GB300 (4 x 8 bucket, K = 8): 3 of 4 words is fastest at both register budgets (3 CTAs
// per SM for the register-held split kernel, 4 for the staged one). The prefetching kernel
// (one or two sources, two tiles in flight) measured fastest with all 4 words split.
constexpr int kSplitWords = 3;
constexpr int kSplitMinCtas = 3;   // k_dequant_reduce_requant_split: 80 registers
constexpr int kStagedMinCtas = 4;  // k_dequant_reduce_requant_staged (KC <= 8): 64 registers

template <int BITS>
struct Geo4 {
  static constexpr int EPL = BITS == 4 ? 32 : 16;  // elements per lane
  static constexpr int ROW = 32 * EPL;
  static constexpr int CTA = kWarps * ROW;
  static constexpr int NP = EPL / 2;                // fp32 pairs per lane
};
constexpr int kEpl5 = 16;
constexpr int kRow5 = 32 * kEpl5;
constexpr int kCta5 = kWarps * kRow5;

// acc += q * s for the 16 code bytes of one source: each term added with one rounding
// (fused multiply-add), in the order the sources are visited. INT4 words k < SPLIT take
// the split conversion (and its pair layout).
template <int BITS, int NWORDS, int SPLIT>
__device__ __forceinline__ void accumulate(f32x2* acc, const uint32_t* w, float s) {
  const f32x2 ss = f2(s, s);
#pragma unroll
  for (int k = 0; k < NWORDS; ++k) {
    if constexpr (BITS == 8) {
      f32x2 q[2];
      int8x4_to_f2(w[k], q);
      acc[2 * k] = f2_fma(q[0], ss, acc[2 * k]);
      acc[2 * k + 1] = f2_fma(q[1], ss, acc[2 * k + 1]);
    } else if (k < SPLIT) {
      f32x2 ev[2], od[2];
      int4x8_to_f2_eo(w[k], ev, od);
      acc[4 * k] = f2_fma(ev[0], ss, acc[4 * k]);
      acc[4 * k + 1] = f2_fma(ev[1], ss, acc[4 * k + 1]);
      acc[4 * k + 2] = f2_fma(od[0], ss, acc[4 * k + 2]);
      acc[4 * k + 3] = f2_fma(od[1], ss, acc[4 * k + 3]);
    } else {
      f32x2 q[4];
      int4x8_to_f2(w[k], q);
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[4 * k + j] = f2_fma(q[j], ss, acc[4 * k + j]);
    }
  }
}

// Sum over K sources at a constant stride, KC loads in flight per chunk. EXACT: K is a
// multiple of KC (no per-source test); LIVE: this lane has data (else it loads nothing).
template <int BITS, int NWORDS, int SPLIT, int KC, bool EXACT>
__device__ __forceinline__ void reduce_sources(f32x2* acc, const uint8_t* cbase, int64_t cstep,
                                               const float* sbase, int64_t sstep, int K, bool live) {
  for (int k0 = 0; k0 < K; k0 += KC) {
    uint32_t raw[KC][NWORDS];
    float s[KC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      if (live && (EXACT || k0 + i < K)) {
        const uint8_t* p = cbase + (k0 + i) * cstep;
        if constexpr (NWORDS == 4) {
          const uint4 v = ld_stream_v4(p);
          raw[i][0] = v.x, raw[i][1] = v.y, raw[i][2 % NWORDS] = v.z, raw[i][3 % NWORDS] = v.w;
        } else {
          const uint2 v = ld_stream_v2(p);
          raw[i][0] = v.x, raw[i][1 % NWORDS] = v.y;
        }
        s[i] = __ldg(sbase + (k0 + i) * sstep);
      } else {
#pragma unroll
        for (int k = 0; k < NWORDS; ++k) raw[i][k] = 0u;
        s[i] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < KC; ++i)
      if (EXACT || k0 + i < K) accumulate<BITS, NWORDS, SPLIT>(acc, raw[i], s[i]);
  }
}

// The end of a K4 tile: block absmax of the lane's EPL sums (across lanes, and across warps
// through `red` for blocks wider than a row of 32 * EPL), block scale, codes, and the stores
// at the receiver's output offsets (codes at byte out_c + e*BITS/8, scales at out_s + e/B).
// A lane's codes are 4 words (st_v4) or 8 words (32 bytes: one 256-bit store when V8).
template <int BITS, int SPLIT, int EPL = Geo4<BITS>::EPL, bool V8 = false>
__device__ __forceinline__ void requant_store(const f32x2* acc, int lane, int warp, int B,
                                              int64_t e, bool valid, int64_t out_c,
                                              int64_t out_s, uint8_t* __restrict__ out_codes,
                                              float* __restrict__ out_scales, float* red) {
  constexpr int NP = EPL / 2, ROW = 32 * EPL, NWORD = EPL * BITS / 32;
  static_assert(NWORD == 4 || NWORD == 8, "a lane stores 16 or 32 code bytes");
  const int log2b = __ffs(B) - 1;
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    float a, b;
    f2_split(acc[j], a, b);
    m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
  }
  if (B <= ROW) {
    m = warp_max(m, B / EPL);
  } else {
    m = warp_max(m, 32);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    const int wpb = B / ROW, w0 = warp & ~(wpb - 1);
    m = red[w0];
    for (int i = 1; i < wpb; ++i) m = fmaxf(m, red[w0 + i]);
  }
  float sc, iv;
  block_scale<BITS>(m, sc, iv);
  if (!valid) return;
  const f32x2 iv2 = f2(iv, iv);
  U8x32 w;
#pragma unroll
  for (int k = 0; k < NWORD; ++k) {
    if constexpr (BITS == 8) {
      const f32x2 q[2] = {round_codes(acc[2 * k], iv2), round_codes(acc[2 * k + 1], iv2)};
      w.w[k] = pack_int8x4(q);
    } else {
      const f32x2 q[4] = {round_codes(acc[4 * k], iv2), round_codes(acc[4 * k + 1], iv2),
                          round_codes(acc[4 * k + 2], iv2), round_codes(acc[4 * k + 3], iv2)};
      w.w[k] = k < SPLIT ? pack_int4x8_eo(q) : pack_int4x8(q);
    }
  }
  uint8_t* dst = out_codes + out_c + e * BITS / 8;
  if constexpr (NWORD == 4)
    st_v4(dst, make_uint4(w.w[0], w.w[1], w.w[2], w.w[3]));
  else
    st_vec32<V8>(dst, w);
  if ((e & (B - 1)) == 0) out_scales[out_s + (e >> log2b)] = sc;
}

// K4. Grid (tile, l - l_begin, n): CTA (x, l, n) owns tile x_begin + x of receiver (n, l) --
// 8 warps x one row each -- so no thread divides to find its work. A launch may cover only
// the receivers whose local index l lies in [l_begin, l_begin + gridDim.y), and only the
// tiles from x_begin on. Blocks wider than a row are reduced across the warps that share
// them through shared memory.
template <int BITS, int KC, bool EXACT, bool FULL, int SPLIT>
__device__ __forceinline__ void drr_tile(const uint8_t* __restrict__ codes,
                                         const float* __restrict__ scales, int64_t E, int64_t C,
                                         int log2b, int M, int l_begin, int x_begin,
                                         uint8_t* __restrict__ out_codes,
                                         float* __restrict__ out_scales, float* red) {
  using G = Geo4<BITS>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = 1 << log2b;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb_in = E * BITS / 8, sc_in = E >> log2b;
  const int64_t cb_out = C * BITS / 8, sc_out = C >> log2b;
  const int64_t e = (static_cast<int64_t>(blockIdx.x) + x_begin) * G::CTA + warp * G::ROW +
                    lane * G::EPL;
  const bool valid = FULL || e < C;  // C is a multiple of the block: whole blocks in or out
  const int64_t idx = static_cast<int64_t>(l) * C + e;  // chunk l of each source
  const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);

  f32x2 acc[G::NP];
#pragma unroll
  for (int j = 0; j < G::NP; ++j) acc[j] = f2(0.0f, 0.0f);
  reduce_sources<BITS, 4, SPLIT, KC, EXACT>(acc, cbase, cb_in, sbase, sc_in, M, valid);

  requant_store<BITS, SPLIT>(acc, lane, warp, B, e, valid, r * cb_out, r * sc_out, out_codes,
                             out_scales, red);
}

template <int BITS, int KC, bool EXACT, int SPLIT>
__device__ __forceinline__ void drr_body(const uint8_t* __restrict__ codes,
                                         const float* __restrict__ scales, int64_t E, int64_t C,
                                         int log2b, int M, int l_begin, int x_begin,
                                         uint8_t* __restrict__ out_codes,
                                         float* __restrict__ out_scales) {
  __shared__ float red[kWarps];
  if ((static_cast<int64_t>(blockIdx.x) + x_begin + 1) * Geo4<BITS>::CTA <= C)  // CTA-uniform
    drr_tile<BITS, KC, EXACT, true, SPLIT>(codes, scales, E, C, log2b, M, l_begin, x_begin,
                                           out_codes, out_scales, red);
  else
    drr_tile<BITS, KC, EXACT, false, SPLIT>(codes, scales, E, C, log2b, M, l_begin, x_begin,
                                            out_codes, out_scales, red);
}

template <int BITS, int KC, bool EXACT>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce_requant(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                             int64_t E, int64_t C, int log2b, int M, int l_begin, int x_begin,
                             uint8_t* __restrict__ out_codes, float* __restrict__ out_scales) {
  drr_body<BITS, KC, EXACT, 0>(codes, scales, E, C, log2b, M, l_begin, x_begin, out_codes,
                               out_scales);
}

template <int KC>
__global__ void __launch_bounds__(kThreads, kSplitMinCtas)
    k_dequant_reduce_requant_split(const uint8_t* __restrict__ codes,
                                   const float* __restrict__ scales, int64_t E, int64_t C,
                                   int log2b, int M, int l_begin, int x_begin,
                                   uint8_t* __restrict__ out_codes,
                                   float* __restrict__ out_scales) {
  drr_body<4, KC, true, kSplitWords>(codes, scales, E, C, log2b, M, l_begin, x_begin, out_codes,
                                     out_scales);
}

// CTA of the staged kernel, which takes INT4 codes only (INT8 codes go to the ring or the
// wide kernel): 4 warps (a 4096-code block is 4 rows, so every block fits one CTA; an INT8
// tile would need 8). Measured on GB300 (4 x 8 bucket, 8 sources): 65.8 us with CTAs of 1,
// 2 or 4 warps against 67.6 us with 8.
template <int BITS>
constexpr int staged_warps() { return BITS == 4 ? 4 : 8; }
template <int BITS, int KC>
constexpr int staged_smem_bytes() { return KC * staged_warps<BITS>() * 32 * 16; }
// CTAs per SM at 64 registers; 16 sources (32 KB of stage per 4-warp CTA): 6 CTAs per SM
template <int BITS, int KC>
constexpr int staged_min_ctas() {
  return KC > 8 ? 3 * 8 / staged_warps<BITS>() : kStagedMinCtas * 8 / staged_warps<BITS>();
}

// K4, INT4 codes, exactly KC (4, 8 or 16) sources per receiver, full tiles only: every
// thread stages its 16 code bytes of each source (32 codes) in shared memory with
// cp.async (the copies do not occupy registers), in two commit groups; the first half of
// the sources is reduced while the second half is still landing. Each thread reads back only
// the slots it filled, and every slot is written once per launch, so no barrier is needed.
// Measured on GB300 (4 x 8 bucket) 68 us against 72 us for the same tile with the codes
// held in registers at 3 CTAs per SM. Grid x counts CTA tiles of staged_warps rows.
template <int BITS, int KC, int SPLIT>
__global__ void __launch_bounds__(staged_warps<BITS>() * 32, staged_min_ctas<BITS, KC>())
    k_dequant_reduce_requant_staged(const uint8_t* __restrict__ codes,
                                    const float* __restrict__ scales, int64_t E, int64_t C,
                                    int log2b, int l_begin, uint8_t* __restrict__ out_codes,
                                    float* __restrict__ out_scales) {
  static_assert(BITS == 4, "INT8 codes take the ring or the wide kernel");
  using G = Geo4<BITS>;
  constexpr int M = KC, H = KC / 2, NT = staged_warps<BITS>() * 32;
  extern __shared__ uint4 stage_mem[];  // [KC][NT], staged_smem_bytes<BITS, KC>()
  uint4(*stage)[NT] = reinterpret_cast<uint4(*)[NT]>(stage_mem);
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb_in = E * BITS / 8, sc_in = E >> log2b;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * (NT / 32 * G::ROW) + warp * G::ROW +
                    lane * G::EPL;
  const int64_t idx = static_cast<int64_t>(l) * C + e;  // chunk l of each source
  const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);
#pragma unroll
  for (int i = 0; i < KC; ++i) {
    cp_async16(&stage[i][threadIdx.x], cbase + i * cb_in);
    if (i == H - 1) cp_async_commit();
  }
  cp_async_commit();
  float s[KC];
#pragma unroll
  for (int i = 0; i < KC; ++i) s[i] = __ldg(sbase + i * sc_in);
  f32x2 acc[G::NP];
#pragma unroll
  for (int j = 0; j < G::NP; ++j) acc[j] = f2(0.0f, 0.0f);
  cp_async_wait<1>();
#pragma unroll
  for (int i = 0; i < KC; ++i) {
    if (i == H) cp_async_wait<0>();
    const uint4 v = stage[i][threadIdx.x];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    accumulate<BITS, 4, SPLIT>(acc, w, s[i]);
  }
  requant_store<BITS, SPLIT>(acc, lane, warp, 1 << log2b, e, true, r * (C * BITS / 8),
                             r * (C >> log2b), out_codes, out_scales, red);
}

// K4 for INT8 codes and exactly KC (1 or 2) sources, whole tiles of 4096 outputs: CTAs of
// 4 warps (a 4096-code block is 4 rows), 32 outputs per lane; each source's 32 code bytes go
// straight into registers (one 256-bit load when the buffers are 32-byte aligned, V8, else
// two 128-bit loads), so a lane's requantisation is spread over twice the outputs of the
// 16-code lanes. Measured on GB300 (topology 1 x 2, 2^28 / 2^30 codes, blocks 64-4096):
// 0.87-0.94 / 0.94-1.01 of the measured copy bandwidth, against 0.57-0.66 / 0.61-0.70 for
// the staged kernel with 16 outputs per lane and 0.67-0.74 for 32 outputs per lane staged
// by two 16-byte cp.async per source.
constexpr int kWide8Warps = 4;
constexpr int kWide8Tile = kWide8Warps * 32 * 32;  // 4096 outputs, = Geo4<8>::CTA

template <int KC, bool V8>
__global__ void __launch_bounds__(kWide8Warps * 32, 8)
    k_dequant_reduce_requant_wide8(const uint8_t* __restrict__ codes,
                                   const float* __restrict__ scales, int64_t E, int64_t C,
                                   int log2b, int l_begin, uint8_t* __restrict__ out_codes,
                                   float* __restrict__ out_scales) {
  constexpr int M = KC, EPL = 32, ROW = 32 * EPL;
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb_in = E, sc_in = E >> log2b;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kWide8Tile + warp * ROW + lane * EPL;
  const int64_t idx = static_cast<int64_t>(l) * C + e;  // chunk l of each source
  const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx;
  const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);
  U8x32 v[KC];
#pragma unroll
  for (int i = 0; i < KC; ++i) v[i] = ld_vec32<V8>(cbase + i * cb_in);
  float s[KC];
#pragma unroll
  for (int i = 0; i < KC; ++i) s[i] = __ldg(sbase + i * sc_in);
  f32x2 acc[EPL / 2];
#pragma unroll
  for (int j = 0; j < EPL / 2; ++j) acc[j] = f2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < KC; ++i) accumulate<8, 8, 0>(acc, v[i].w, s[i]);
  requant_store<8, 0, EPL, V8>(acc, lane, warp, 1 << log2b, e, true, r * C, r * (C >> log2b),
                               out_codes, out_scales, red);
}

// K4 for INT4 codes and exactly KC (1 or 2) sources. With so few terms per output the
// requantisation and the load latency dominate, so each CTA (4 warps) takes two tiles of
// 4096 outputs and loads both tiles' codes (16 bytes per source per lane) into registers
// before converting the first; every code word takes the split conversion. A CTA covers
// one 8-warp tile of Geo4<4> (8192 outputs). Measured on GB300 (topology 1 x 2, 2^28 / 2^30
// codes, blocks 64-4096): 0.58-0.68 / 0.63-0.74 of the measured copy bandwidth, against
// 0.42-0.49 / 0.43-0.52 for the staged kernel (one tile per CTA); three or four tiles per
// CTA measured no better than two.
constexpr int kPrefetchWarps = 4;
constexpr int kPrefetchTile = kPrefetchWarps * 1024;  // outputs per tile; two per CTA

template <int KC>
__global__ void __launch_bounds__(kPrefetchWarps * 32, 8)
    k_dequant_reduce_requant_prefetch(const uint8_t* __restrict__ codes,
                                      const float* __restrict__ scales, int64_t E, int64_t C,
                                      int log2b, int l_begin, uint8_t* __restrict__ out_codes,
                                      float* __restrict__ out_scales) {
  using G = Geo4<4>;
  constexpr int M = KC;
  __shared__ float red[2][kWarps];  // one row per tile: blocks wider than a row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb_in = E / 2, sc_in = E >> log2b;
  const int64_t e0 =
      static_cast<int64_t>(blockIdx.x) * (2 * kPrefetchTile) + warp * G::ROW + lane * G::EPL;
  const int64_t idx0 = static_cast<int64_t>(l) * C + e0;  // chunk l of each source
  const uint8_t* cbase = codes + static_cast<int64_t>(n) * M * cb_in + idx0 / 2;
  const float* sbase = scales + static_cast<int64_t>(n) * M * sc_in;
  uint4 v[2][KC];
  float s[2][KC];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      v[t][i] = ld_stream_v4(cbase + i * cb_in + t * (kPrefetchTile / 2));
      s[t][i] = __ldg(sbase + i * sc_in + ((idx0 + t * kPrefetchTile) >> log2b));
    }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    f32x2 acc[G::NP];
#pragma unroll
    for (int j = 0; j < G::NP; ++j) acc[j] = f2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      const uint32_t w[4] = {v[t][i].x, v[t][i].y, v[t][i].z, v[t][i].w};
      accumulate<4, 4, 4>(acc, w, s[t][i]);
    }
    requant_store<4, 4>(acc, lane, warp, 1 << log2b, e0 + t * kPrefetchTile, true, r * (C / 2),
                        r * (C >> log2b), out_codes, out_scales, red[t]);
  }
}

// ---------------------------------------------------------------------------------
// K4 for INT8 codes and 3 or more sources: a bulk-copy ring. One CTA per SM; 16 consumer
// warps and one producer
// warp. A unit is 8192 consecutive outputs of one receiver (16 warps x 32 lanes x 16
// codes); the units are dealt to the CTAs round robin. The producer streams each unit's
// sources, KC at a time, into a ring of NS shared-memory stages with cp.async.bulk (one
// 8 KB copy per source: 16 warps x 512 B) plus the matching block scales, each stage
// completed by an mbarrier; the consumers read their 16 code bytes per source from the
// stage, accumulate exactly as the other K4 kernels do, release the stage (a second
// mbarrier) and requantise. INT8 codes carry half the terms per byte of INT4 codes, so
// this kernel is bound by memory, and the ring keeps the loads in flight while the
// consumers compute: measured on GB300 at 2^30 INT8 codes, K = 8 / 16, 184 / 166 us
// against 205 / 213 us for the per-CTA staged kernel. (For INT4 codes the same ring
// measured 80-88 us on the 4 x 8 bucket against 68 us for the staged kernel: there the
// conversion work needs the 32 warps per SM that a producer warp would not leave room
// for.)
//
// Every wait is bounded (kRingWaitNs); a wait that runs out sets a bit of g_zpp_fault,
// and the warp continues without waiting (its results are then unspecified), so the
// kernel always ends. Before the CTA exits the producer waits (bounded) for the copies it
// issued that no consumer waited for.
// ---------------------------------------------------------------------------------
__device__ unsigned int g_zpp_fault;

constexpr unsigned long long kRingWaitNs = 1000000000ull;  // 1 s
constexpr int kRingConsumers = 16;
constexpr int kRingThreads = (kRingConsumers + 1) * 32;
constexpr int kRingEpl = 16;                           // INT8 codes per lane
constexpr int kRingRow = 32 * kRingEpl;                // 512 outputs per warp
constexpr int kRingTile = kRingConsumers * kRingRow;   // 8192 outputs per unit
constexpr int kRingSrcBytes = kRingTile;               // code bytes per source per unit
constexpr int kRingScaleSlots = kRingTile / 64;        // scales per source per unit (block >= 64)

template <int KC>
struct RingGeo {
  static constexpr int STAGES = KC == 8 ? 3 : (KC == 4 ? 6 : (KC == 2 ? 12 : 24));
  static constexpr int CODES = STAGES * KC * kRingSrcBytes;
  static constexpr int SCALES = STAGES * KC * kRingScaleSlots * 4;
  static constexpr int SMEM = CODES + SCALES + 2 * STAGES * 8 + 2 * 32 * 4;
};

// Grid: persistent CTAs. Units u = blockIdx.x, blockIdx.x + gridDim.x, ... < U, where
// U = N * (l_end - l_begin) * T, T = ceil(C / kRingTile); unit u is tile x = u % T of the
// receiver with index u / T among those with local index in [l_begin, l_end).
template <int KC>
__global__ void __launch_bounds__(kRingThreads, 1)
    k_dequant_reduce_requant_ring8(const uint8_t* __restrict__ codes,
                                   const float* __restrict__ scales, int64_t E, int64_t C,
                                   int log2b, int N, int M, int l_begin, int l_end,
                                   bool scales_bulk, uint8_t* __restrict__ out_codes,
                                   float* __restrict__ out_scales) {
  using G = RingGeo<KC>;
  constexpr int NS = G::STAGES;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* st_codes = smem;                                         // [NS][KC][kRingSrcBytes]
  float* st_scales = reinterpret_cast<float*>(smem + G::CODES);     // [NS][KC][kRingScaleSlots]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::CODES + G::SCALES);
  uint64_t* empty = full + NS;
  float* red = reinterpret_cast<float*>(empty + NS);  // [2][32] per-warp absmax

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1 + 32);  // the producer's expect_tx arrival + 32 lanes' scale copies
      mbar_init(&empty[s], kRingConsumers);
    }
    mbar_init_fence();
  }
  __syncthreads();

  const int L = l_end - l_begin;
  const uint32_t T = static_cast<uint32_t>((C + kRingTile - 1) / kRingTile);
  const uint32_t U = static_cast<uint32_t>(N) * L * T;
  const int groups = M / KC;

  if (warp == kRingConsumers) {  // producer
    const int64_t cb_in = E, sc_in = E >> log2b;  // INT8: one code byte per element
    int s = 0;
    unsigned phase = 1;  // a fresh barrier counts its (virtual) previous phase as complete
    bool ok = true;
    uint32_t issued = 0;
    for (uint32_t u = blockIdx.x; u < U && ok; u += gridDim.x) {
      const uint32_t rho = u / T, x = u - rho * T;
      const int n = static_cast<int>(rho / L), l = l_begin + static_cast<int>(rho - n * L);
      const int64_t e0 = static_cast<int64_t>(x) * kRingTile;
      const int valid = static_cast<int>(C - e0 < kRingTile ? C - e0 : kRingTile);
      const int64_t idx = static_cast<int64_t>(l) * C + e0;  // chunk l of each source
      const uint8_t* csrc = codes + static_cast<int64_t>(n) * M * cb_in + idx;
      const float* ssrc = scales + static_cast<int64_t>(n) * M * sc_in + (idx >> log2b);
      const int nsc = valid >> log2b;  // whole blocks: C and e0 are multiples of the block
      // the unit's scales of one source: one bulk copy when they span whole 16-byte
      // groups at 16-byte aligned addresses, else one 4-byte copy each
      const bool bulk_sc = scales_bulk && (nsc & 3) == 0;
      for (int g = 0; g < groups; ++g) {
        if (!mbar_try_wait(&empty[s], phase) && !mbar_wait_bounded(&empty[s], phase, kRingWaitNs)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], (static_cast<unsigned>(valid) +
                                           (bulk_sc ? 4u * nsc : 0u)) * KC);
#pragma unroll
          for (int i = 0; i < KC; ++i) {
            bulk_load(st_codes + (s * KC + i) * kRingSrcBytes,
                      csrc + static_cast<int64_t>(g * KC + i) * cb_in, static_cast<unsigned>(valid),
                      &full[s]);
            if (bulk_sc)
              bulk_load(st_scales + (s * KC + i) * kRingScaleSlots,
                        ssrc + static_cast<int64_t>(g * KC + i) * sc_in, 4u * nsc, &full[s]);
          }
        }
        if (!bulk_sc)
          for (int j = lane; j < KC * nsc; j += 32) {
            const int i = j / nsc, b = j - i * nsc;
            cp_async4(st_scales + (s * KC + i) * kRingScaleSlots + b,
                      ssrc + static_cast<int64_t>(g * KC + i) * sc_in + b);
          }
        cp_async_arrive_noinc(&full[s]);  // counts even with no copies of its own
        ++issued;
        if (++s == NS) s = 0, phase ^= 1u;
      }
    }
    if (!ok && lane == 0) atomicOr(&g_zpp_fault, 1u);
    // The stages issued last may not have been waited for by any consumer (after a
    // timeout): wait for them, bounded, before the CTA may exit.
    unsigned dphase = phase ^ 1u;
    int ds = s;
    for (uint32_t d = 0; d < static_cast<uint32_t>(NS) && d < issued; ++d) {
      if (--ds < 0) ds = NS - 1, dphase ^= 1u;
      if (!mbar_try_wait(&full[ds], dphase)) mbar_wait_bounded(&full[ds], dphase, kRingWaitNs);
    }
    return;
  }

  const int B = 1 << log2b;
  const int lane_e = warp * kRingRow + lane * kRingEpl;  // output offset within a unit
  const int sidx = lane_e >> log2b;
  const int lane_c = (warp * 32 + lane) * 16;
  int s = 0;
  unsigned phase = 0;
  int ub = 0;
  bool alive = true;  // false once a wait ran out: no more waits, results unspecified
  for (uint32_t u = blockIdx.x; u < U; u += gridDim.x, ub ^= 1) {
    f32x2 acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = f2(0.0f, 0.0f);
    for (int g = 0; g < groups; ++g) {
      if (!mbar_try_wait(&full[s], phase) && alive &&
          !mbar_wait_bounded(&full[s], phase, kRingWaitNs)) {
        alive = false;
        if (lane == 0) atomicOr(&g_zpp_fault, 2u);
      }
      const uint8_t* cs = st_codes + s * (KC * kRingSrcBytes) + lane_c;
      const float* ss = st_scales + s * (KC * kRingScaleSlots) + sidx;
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(cs + i * kRingSrcBytes);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        accumulate<8, 4, 0>(acc, w, ss[i * kRingScaleSlots]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == NS) s = 0, phase ^= 1u;
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a, b;
      f2_split(acc[j], a, b);
      m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
    }
    if (B <= kRingRow) {
      m = warp_max(m, B / kRingEpl);
    } else {  // a block spans B / kRingRow consumer warps of the unit
      m = warp_max(m, 32);
      if (lane == 0) red[ub * 32 + warp] = m;
      named_barrier(1, kRingConsumers * 32);
      const int wpb = B / kRingRow, w0 = warp & ~(wpb - 1);
      m = red[ub * 32 + w0];
      for (int i = 1; i < wpb; ++i) m = fmaxf(m, red[ub * 32 + w0 + i]);
    }
    float sc, iv;
    block_scale<8>(m, sc, iv);
    const uint32_t rho = u / T, x = u - rho * T;
    const int n = static_cast<int>(rho / L), l = l_begin + static_cast<int>(rho - n * L);
    const int64_t e = static_cast<int64_t>(x) * kRingTile + lane_e;
    if (e < C) {  // C is a multiple of the block: whole blocks are in or out
      const f32x2 iv2 = f2(iv, iv);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const f32x2 q[2] = {round_codes(acc[2 * k], iv2), round_codes(acc[2 * k + 1], iv2)};
        w[k] = pack_int8x4(q);
      }
      const int64_t o = (static_cast<int64_t>(n) * M + l) * C + e;  // receiver r = n*M + l
      st_v4(out_codes + o, make_uint4(w[0], w[1], w[2], w[3]));
      if ((e & (B - 1)) == 0) out_scales[o >> log2b] = sc;
    }
  }
}

// Diagnostic: a wait on an mbarrier that nothing completes, bounded by limit_ns; sets bit 4
// of g_zpp_fault when it runs out (it always does). Exercises the bounded wait and the
// fault word on the device without a fault of any kind.
__global__ void k_wait_selftest(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_try_wait(&bar, 0) && !mbar_wait_bounded(&bar, 0, limit_ns))
    atomicOr(&g_zpp_fault, 4u);
}

// K5. Grid (tile, l, n) as for K4. A lane owns 16 consecutive outputs of its receiver's
// slice: the sums, multiplied by post_scale (1 for the plain sum, 1/W for the average; one
// fp32 rounding), are written with 256-bit stores as fp32 (each store a full 32-byte
// sector) or rounded to fp16 / bf16. S is the slice each receiver owns and C the length of
// one hop-1 output; the N sources of receiver (n, l) are the hop-1 outputs of ranks
// (n', l), at a stride of M outputs, from which it reads slice n.
template <int BITS, int KC, bool EXACT, typename OT, bool V8>
__global__ void __launch_bounds__(kThreads)
    k_dequant_reduce(const uint8_t* __restrict__ codes, const float* __restrict__ scales, int64_t S,
                     int64_t C, int log2b, int N, int M, int l_begin, float post_scale,
                     void* __restrict__ out) {
  constexpr int NW = BITS == 8 ? 4 : 2;  // code words per lane per source
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb = C * BITS / 8, sc = C >> log2b;  // per hop-1 rank
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kCta5 + warp * kRow5 + lane * kEpl5;
  if (e >= S) return;  // no barrier in this kernel
  const int64_t idx = static_cast<int64_t>(n) * S + e;  // slice n of each hop-1 output
  const uint8_t* cbase = codes + static_cast<int64_t>(l) * cb + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(l) * sc + (idx >> log2b);

  f32x2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = f2(0.0f, 0.0f);
  reduce_sources<BITS, NW, 0, KC, EXACT>(acc, cbase, static_cast<int64_t>(M) * cb, sbase,
                                         static_cast<int64_t>(M) * sc, N, true);
  const f32x2 ps = f2(post_scale, post_scale);
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) f2_split(f2_mul(acc[j], ps), v[2 * j], v[2 * j + 1]);
  store16<OT, V8>(out, r * S + e, v);
}

// K5 with exactly KC sources (N == KC in {1, 2, 4, 8}): every source's code words and scale
// are loaded before the first sum, with no source loop. When the words in flight are at
// most 8 per lane (INT4 with up to 4 sources, INT8 with up to 2) the kernel fits 32
// registers, so 8 CTAs (64 warps) per SM keep the most loads in flight: measured on GB300
// (4 x 8 bucket, N = 4) 14.8 us against 18.5 us for the looping kernel at 40 registers.
template <int BITS, int KC>
constexpr int dr_min_ctas() { return KC * (BITS == 8 ? 4 : 2) <= 8 ? 8 : 1; }

template <int BITS, int KC, typename OT, bool V8>
__global__ void __launch_bounds__(kThreads, dr_min_ctas<BITS, KC>())
    k_dequant_reduce_all(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                         int64_t S, int64_t C, int log2b, int M, int l_begin, float post_scale,
                         void* __restrict__ out) {
  constexpr int NW = BITS == 8 ? 4 : 2;  // code words per lane per source
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = l_begin + static_cast<int>(blockIdx.y), n = blockIdx.z;
  const int64_t r = static_cast<int64_t>(n) * M + l;
  const int64_t cb = C * BITS / 8, sc = C >> log2b;  // per hop-1 rank
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kCta5 + warp * kRow5 + lane * kEpl5;
  if (e >= S) return;  // no barrier in this kernel
  const int64_t idx = static_cast<int64_t>(n) * S + e;  // slice n of each hop-1 output
  const uint8_t* cbase = codes + static_cast<int64_t>(l) * cb + idx * BITS / 8;
  const float* sbase = scales + static_cast<int64_t>(l) * sc + (idx >> log2b);
  const int64_t cstep = static_cast<int64_t>(M) * cb, sstep = static_cast<int64_t>(M) * sc;
  uint32_t w[KC][NW];
  float s[KC];
#pragma unroll
  for (int i = 0; i < KC; ++i) {
    if constexpr (NW == 4) {
      const uint4 v = ld_stream_v4(cbase + i * cstep);
      w[i][0] = v.x, w[i][1] = v.y, w[i][2 % NW] = v.z, w[i][3 % NW] = v.w;
    } else {
      const uint2 v = ld_stream_v2(cbase + i * cstep);
      w[i][0] = v.x, w[i][1 % NW] = v.y;
    }
    s[i] = __ldg(sbase + i * sstep);
  }
  f32x2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = f2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < KC; ++i) accumulate<BITS, NW, 0>(acc, w[i], s[i]);
  const f32x2 ps = f2(post_scale, post_scale);
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) f2_split(f2_mul(acc[j], ps), v[2 * j], v[2 * j + 1]);
  store16<OT, V8>(out, r * S + e, v);
}

static int chunk_for(int k) { return k >= 8 ? 8 : (k > 2 ? 4 : (k == 2 ? 2 : 1)); }

// `full`: the number of whole 8-warp tiles (Geo4<BITS>::CTA outputs) per receiver
template <int BITS, int KC, int SPLIT>
static cudaError_t run_staged(const uint8_t* c, const float* scales, int64_t E, int64_t C,
                              int log2b, int lb, int64_t full, unsigned ny, unsigned nz,
                              uint8_t* oc, float* out_scales, cudaStream_t s) {
  constexpr int smem = staged_smem_bytes<BITS, KC>();
  constexpr int NW = staged_warps<BITS>();
  auto kern = k_dequant_reduce_requant_staged<BITS, KC, SPLIT>;
  if constexpr (smem > 48 * 1024) {  // above the default dynamic shared-memory limit
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<dim3(static_cast<unsigned>(full * (kWarps / NW)), ny, nz), NW * 32, smem, s>>>(
      c, scales, E, C, log2b, lb, oc, out_scales);
  return cudaGetLastError();
}

// INT4 codes, 3 or more sources, in chunks of KC (4 or 8): the staged kernel when one chunk
// holds every source (M = KC, or M = 16 as one stage of 16), else the split / register kernels.
template <int BITS, int KC>
static cudaError_t run_drr(const void* codes, const float* scales, int64_t E, int64_t C, int log2b,
                           int N, int M, int lb, int le, void* out_codes, float* out_scales,
                           cudaStream_t s) {
  static_assert(BITS == 4 && KC >= 4, "one or two sources and INT8 codes have their own kernels");
  constexpr int CTA = Geo4<BITS>::CTA;
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  uint8_t* oc = static_cast<uint8_t*>(out_codes);
  const unsigned ny = static_cast<unsigned>(le - lb), nz = static_cast<unsigned>(N);
  if constexpr (KC >= 2) {
    if (M == KC || (KC == 8 && M == 16)) {  // one stage of sources on the full tiles, then the tail
      constexpr int SPLIT = BITS == 4 && KC >= 4 ? kSplitWords : 0;
      const int64_t full = C / CTA;
      cudaError_t err = cudaSuccess;
      if (full > 0) {
        if (M == KC)
          err = run_staged<BITS, KC, SPLIT>(c, scales, E, C, log2b, lb, full, ny, nz, oc,
                                            out_scales, s);
        else if constexpr (KC == 8)  // M == 16
          err = run_staged<BITS, 16, SPLIT>(c, scales, E, C, log2b, lb, full, ny, nz, oc,
                                            out_scales, s);
      }
      if (err != cudaSuccess) return err;
      if (C % CTA != 0) {
        if constexpr (BITS == 4 && KC >= 4)
          k_dequant_reduce_requant_split<KC><<<dim3(1, ny, nz), kThreads, 0, s>>>(
              c, scales, E, C, log2b, M, lb, static_cast<int>(full), oc, out_scales);
        else
          k_dequant_reduce_requant<BITS, KC, true><<<dim3(1, ny, nz), kThreads, 0, s>>>(
              c, scales, E, C, log2b, M, lb, static_cast<int>(full), oc, out_scales);
      }
      return cudaGetLastError();
    }
  }
  const dim3 grid(tile_grid(C, CTA), ny, nz);
  if (M % KC != 0)
    k_dequant_reduce_requant<BITS, KC, false><<<grid, kThreads, 0, s>>>(c, scales, E, C, log2b, M,
                                                                        lb, 0, oc, out_scales);
  else if constexpr (BITS == 4 && KC >= 4)
    k_dequant_reduce_requant_split<KC><<<grid, kThreads, 0, s>>>(c, scales, E, C, log2b, M, lb, 0,
                                                                 oc, out_scales);
  else
    k_dequant_reduce_requant<BITS, KC, true><<<grid, kThreads, 0, s>>>(c, scales, E, C, log2b, M,
                                                                       lb, 0, oc, out_scales);
  return cudaGetLastError();
}

template <int BITS, int KC, typename OT>
static cudaError_t run_dr(const void* codes, const float* scales, int64_t S, int64_t C, int log2b,
                          int N, int M, int lb, int le, int nz, float post_scale, void* out,
                          cudaStream_t s) {
  const dim3 grid(tile_grid(S, kCta5), le - lb, nz);
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  // out + (r*S + e) elements stays 32-byte aligned when out is: S and e are multiples of 16
  const bool v8 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
  if (N == KC) {  // one chunk: every source loaded up front
    if (v8)
      k_dequant_reduce_all<BITS, KC, OT, true><<<grid, kThreads, 0, s>>>(c, scales, S, C, log2b, M,
                                                                         lb, post_scale, out);
    else
      k_dequant_reduce_all<BITS, KC, OT, false><<<grid, kThreads, 0, s>>>(c, scales, S, C, log2b,
                                                                          M, lb, post_scale, out);
  } else if (N % KC == 0) {
    if (v8)
      k_dequant_reduce<BITS, KC, true, OT, true><<<grid, kThreads, 0, s>>>(c, scales, S, C, log2b,
                                                                          N, M, lb, post_scale,
                                                                          out);
    else
      k_dequant_reduce<BITS, KC, true, OT, false><<<grid, kThreads, 0, s>>>(c, scales, S, C, log2b,
                                                                           N, M, lb, post_scale,
                                                                           out);
  } else {
    if (v8)
      k_dequant_reduce<BITS, KC, false, OT, true><<<grid, kThreads, 0, s>>>(c, scales, S, C, log2b,
                                                                           N, M, lb, post_scale,
                                                                           out);
    else
      k_dequant_reduce<BITS, KC, false, OT, false><<<grid, kThreads, 0, s>>>(c, scales, S, C,
                                                                            log2b, N, M, lb,
                                                                            post_scale, out);
  }
  return cudaGetLastError();
}

template <int KC>
static cudaError_t run_ring8(const void* codes, const float* scales, int64_t E, int64_t C,
                            int log2b, int N, int M, int lb, int le, void* out_codes,
                            float* out_scales, cudaStream_t s) {
  auto kern = k_dequant_reduce_requant_ring8<KC>;
  constexpr int smem = RingGeo<KC>::SMEM;
  // per-device set-up, done once: the dynamic shared-memory limit and the SM count
  constexpr int kMaxDevices = 64;
  static int sms_of[kMaxDevices];  // 0: not set up yet
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int sms = dev < kMaxDevices ? sms_of[dev] : 0;
  if (sms == 0) {
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err;
    if (dev < kMaxDevices) sms_of[dev] = sms;
  }
  const int64_t T = (C + kRingTile - 1) / kRingTile;
  const int64_t U = static_cast<int64_t>(N) * (le - lb) * T;
  const unsigned grid = static_cast<unsigned>(U < sms ? U : sms);
  // scale rows start on 16-byte boundaries: per-source stride, chunk offsets and unit
  // offsets all whole groups of 4 scales, and the array itself 16-byte aligned
  const int64_t sc_in = E >> log2b;
  const bool scales_bulk = (reinterpret_cast<uintptr_t>(scales) & 15) == 0 && sc_in % 4 == 0 &&
                           (C >> log2b) % 4 == 0 && (kRingTile >> log2b) % 4 == 0;
  kern<<<grid, kRingThreads, smem, s>>>(static_cast<const uint8_t*>(codes), scales, E, C, log2b,
                                        N, M, lb, le, scales_bulk,
                                        static_cast<uint8_t*>(out_codes), out_scales);
  return cudaGetLastError();
}

// INT4, M = KC (1 or 2) sources: the whole 8192-output tiles through the prefetching kernel,
// a ragged last tile through the register kernel at that tile offset.
template <int KC>
static cudaError_t run_prefetch(const void* codes, const float* scales, int64_t E, int64_t C,
                               int log2b, int N, int lb, int le, void* out_codes,
                               float* out_scales, cudaStream_t s) {
  static_assert(2 * kPrefetchTile == Geo4<4>::CTA, "the tail kernel's tile offset counts CTAs");
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  uint8_t* oc = static_cast<uint8_t*>(out_codes);
  const unsigned ny = static_cast<unsigned>(le - lb), nz = static_cast<unsigned>(N);
  const int64_t full = C / Geo4<4>::CTA;
  if (full > 0) {
    k_dequant_reduce_requant_prefetch<KC>
        <<<dim3(static_cast<unsigned>(full), ny, nz), kPrefetchWarps * 32, 0, s>>>(
            c, scales, E, C, log2b, lb, oc, out_scales);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (C % Geo4<4>::CTA != 0)
    k_dequant_reduce_requant<4, KC, true><<<dim3(1, ny, nz), kThreads, 0, s>>>(
        c, scales, E, C, log2b, KC, lb, static_cast<int>(full), oc, out_scales);
  return cudaGetLastError();
}

// INT8, M = KC (1 or 2) sources: the whole 4096-output tiles through the wide kernel, a ragged
// last tile through the register kernel at that tile offset.
template <int KC>
static cudaError_t run_wide8(const void* codes, const float* scales, int64_t E, int64_t C,
                            int log2b, int N, int lb, int le, void* out_codes, float* out_scales,
                            cudaStream_t s) {
  static_assert(kWide8Tile == Geo4<8>::CTA, "the tail kernel's tile offset counts wide tiles");
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  uint8_t* oc = static_cast<uint8_t*>(out_codes);
  const unsigned ny = static_cast<unsigned>(le - lb), nz = static_cast<unsigned>(N);
  const int64_t full = C / kWide8Tile;
  if (full > 0) {
    // every lane's 32 code bytes start on a 32-byte boundary when both bases do (E and C
    // are multiples of the block, so of 64)
    const bool v8 = ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(out_codes)) &
                     31) == 0;
    const dim3 grid(static_cast<unsigned>(full), ny, nz);
    if (v8)
      k_dequant_reduce_requant_wide8<KC, true><<<grid, kWide8Warps * 32, 0, s>>>(
          c, scales, E, C, log2b, lb, oc, out_scales);
    else
      k_dequant_reduce_requant_wide8<KC, false><<<grid, kWide8Warps * 32, 0, s>>>(
          c, scales, E, C, log2b, lb, oc, out_scales);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (C % kWide8Tile != 0)
    k_dequant_reduce_requant<8, KC, true><<<dim3(1, ny, nz), kThreads, 0, s>>>(
        c, scales, E, C, log2b, KC, lb, static_cast<int>(full), oc, out_scales);
  return cudaGetLastError();
}

template <int BITS>
static cudaError_t drr_bits(const void* c, const float* sc, int64_t E, int64_t C, int log2b, int N,
                            int M, int lb, int le, void* oc, float* os, cudaStream_t s) {
  // INT8 with 3 or more sources: the bulk-copy ring (sources in groups of KC). With one or
  // two sources the requantisation dominates: the wide kernel (32 outputs per lane, codes
  // in registers) spreads it over the most outputs (2^30 codes, K = 2: 246-251 us, against
  // 389 us staged and 489 us in the ring).
  if constexpr (BITS == 8) {
    if (M > 2) {
      if (M % 8 == 0) return run_ring8<8>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
      if (M % 4 == 0) return run_ring8<4>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
      if (M % 2 == 0) return run_ring8<2>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
      return run_ring8<1>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
    }
    if (M == 2) return run_wide8<2>(c, sc, E, C, log2b, N, lb, le, oc, os, s);
    return run_wide8<1>(c, sc, E, C, log2b, N, lb, le, oc, os, s);
  } else {
    // INT4 with one or two sources: two tiles per CTA, both loaded before the first is
    // converted (2^30 codes, K = 2: 181-189 us against 257-274 us staged)
    if (M == 2) return run_prefetch<2>(c, sc, E, C, log2b, N, lb, le, oc, os, s);
    if (M == 1) return run_prefetch<1>(c, sc, E, C, log2b, N, lb, le, oc, os, s);
    switch (chunk_for(M)) {
      case 8: return run_drr<BITS, 8>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
      default: return run_drr<BITS, 4>(c, sc, E, C, log2b, N, M, lb, le, oc, os, s);
    }
  }
}

template <int BITS, typename OT>
static cudaError_t dr_bits(const void* c, const float* sc, int64_t S, int64_t C, int log2b, int N,
                           int M, int lb, int le, int nz, float ps, void* out, cudaStream_t s) {
  switch (chunk_for(N)) {
    case 8: return run_dr<BITS, 8, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s);
    case 4: return run_dr<BITS, 4, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s);
    case 2: return run_dr<BITS, 2, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s);
    default: return run_dr<BITS, 1, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s);
  }
}

template <typename OT>
static cudaError_t dr_out(const void* c, const float* sc, int64_t S, int64_t C, int log2b, int bits,
                          int N, int M, int lb, int le, int nz, float ps, void* out,
                          cudaStream_t s) {
  return bits == 8 ? dr_bits<8, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s)
                   : dr_bits<4, OT>(c, sc, S, C, log2b, N, M, lb, le, nz, ps, out, s);
}

cudaError_t launch_dequant_reduce_requant(const void* codes, const float* scales, int64_t E,
                                          int64_t C, int block, int bits, int N, int M,
                                          int l_begin, int l_end, void* out_codes,
                                          float* out_scales, cudaStream_t s) {
  const int log2b = __builtin_ctz(static_cast<unsigned>(block));
  return bits == 8 ? drr_bits<8>(codes, scales, E, C, log2b, N, M, l_begin, l_end, out_codes,
                                 out_scales, s)
                   : drr_bits<4>(codes, scales, E, C, log2b, N, M, l_begin, l_end, out_codes,
                                 out_scales, s);
}

cudaError_t read_device_fault(unsigned* flags, bool clear) {
  cudaError_t err = cudaMemcpyFromSymbol(flags, g_zpp_fault, sizeof(unsigned));
  if (err != cudaSuccess || !clear) return err;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_zpp_fault, &zero, sizeof(unsigned));
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_dequant_reduce(const void* codes, const float* scales, int64_t S, int64_t C,
                                  int block, int bits, int N, int M, int l_begin, int l_end,
                                  int nz, float post_scale, void* out, int out_kind,
                                  cudaStream_t s) {
  const int log2b = __builtin_ctz(static_cast<unsigned>(block));
  if (out_kind == 0)
    return dr_out<OutF16>(codes, scales, S, C, log2b, bits, N, M, l_begin, l_end, nz, post_scale,
                          out, s);
  if (out_kind == 1)
    return dr_out<OutBF16>(codes, scales, S, C, log2b, bits, N, M, l_begin, l_end, nz, post_scale,
                           out, s);
  return dr_out<OutF32>(codes, scales, S, C, log2b, bits, N, M, l_begin, l_end, nz, post_scale,
                        out, s);
}

}  // namespace zpp
