// zpp_device.cuh -- device-side building blocks shared by the sm_103a kernels:
// 256-bit global vector accesses, 16-bit float unpacking, absmax, and the block
// quantiser's per-element arithmetic.
//
// Numerics: every fp32 operation uses an explicitly rounded intrinsic (__fmul_rn,
// __fadd_rn, __fdiv_rn, __float2int_rn), so no multiply-add is ever contracted into an
// FMA and each division is the IEEE one; the build also passes -fmad=false and keeps
// denormals (no -ftz).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace zpp {

constexpr int kThreads = 256;  // threads per CTA for every kernel (8 warps)
constexpr int kWarps = kThreads / 32;

struct alignas(32) U8x32 {  // 32 bytes as eight 32-bit words
  uint32_t w[8];
};

// ---------------------------------------------------------------------------------
// Global memory vector accesses. Loads of data read exactly once take the read-only
// path without L1 allocation.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ U8x32 ld_stream_v8(const void* p) {
  U8x32 r;
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_b32(const void* p) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v8(void* p, const U8x32& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------------------------
// 16-bit float formats. Tag types select fp16 / bf16 at compile time.
// ---------------------------------------------------------------------------------
struct F16 {};
struct BF16 {};

// Two packed 16-bit values -> two floats (exact).
__device__ __forceinline__ float2 unpack2(uint32_t w, F16) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
__device__ __forceinline__ float2 unpack2(uint32_t w, BF16) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// One 16-bit magnitude pattern -> float (exact).
__device__ __forceinline__ float bits16_to_float(uint32_t b, F16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}
__device__ __forceinline__ float bits16_to_float(uint32_t b, BF16) { return __uint_as_float(b << 16); }

// Two floats -> two packed 16-bit values, round to nearest even.
__device__ __forceinline__ uint32_t pack2(float a, float b, F16) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, BF16) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Largest magnitude among the 16-bit values of `nw` words, as a 16-bit pattern. For
// finite fp16/bf16 values the sign-cleared bit patterns order exactly like |x|, so
// the maximum is taken on integers, two lanes per instruction.
template <int NW>
__device__ __forceinline__ uint32_t absmax_bits16(const uint32_t* w) {
  uint32_t m = w[0] & 0x7fff7fffu;
#pragma unroll
  for (int i = 1; i < NW; ++i) m = __vmaxu2(m, w[i] & 0x7fff7fffu);
  return max(m & 0xffffu, m >> 16);
}

// ---------------------------------------------------------------------------------
// The block quantiser: scale and inverse of one block, then per-element codes.
// ---------------------------------------------------------------------------------
template <int BITS>
struct QParams {
  static constexpr int qmax = (1 << (BITS - 1)) - 1;
};

// scale = amax / qmax, inv = qmax / amax (IEEE divisions); a block whose inverse is not
// finite (amax == 0, or amax so small that qmax / amax overflows) gets scale 0 and
// inverse 0, which makes every code 0.
template <int BITS>
__device__ __forceinline__ void block_scale(float amax, float& scale, float& inv) {
  const float qm = static_cast<float>(QParams<BITS>::qmax);
  inv = __fdiv_rn(qm, amax);
  scale = __fdiv_rn(amax, qm);
  if (!isfinite(inv)) {
    inv = 0.0f;
    scale = 0.0f;
  }
}

// q = clamp(rint_even(x * inv), -qmax, qmax)
template <int BITS>
__device__ __forceinline__ int quantize(float x, float inv) {
  int q = __float2int_rn(__fmul_rn(x, inv));
  q = max(q, -QParams<BITS>::qmax);
  return min(q, QParams<BITS>::qmax);
}

// Pack eight signed codes: INT8 -> two words (byte i = code i); INT4 -> one word
// (nibble i = code i, so element 2k is the low nibble of byte k).
__device__ __forceinline__ uint2 pack8_int8(const int* q) {
  uint2 r;
  r.x = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)q[3] << 24);
  r.y = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | ((uint32_t)q[7] << 24);
  return r;
}
__device__ __forceinline__ uint32_t pack8_int4(const int* q) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) r |= (static_cast<uint32_t>(q[i]) & 0xfu) << (4 * i);
  return r;
}

// Signed code i of a packed word (sign-extended by arithmetic shifts).
__device__ __forceinline__ int code_int8(uint32_t w, int i) {
  return static_cast<int>(w << (24 - 8 * i)) >> 24;
}
__device__ __forceinline__ int code_int4(uint32_t w, int i) {
  return static_cast<int>(w << (28 - 4 * i)) >> 28;
}

__device__ __forceinline__ float warp_max(float v, int width) {
  for (int off = width >> 1; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v, int width) {
  for (int off = width >> 1; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

}  // namespace zpp
