// zpp_device.cuh -- device-side building blocks shared by the sm_103a kernels:
// 256-bit global vector accesses, 16-bit float unpacking, absmax, and the block
// quantiser's per-element arithmetic.
//
// Numerics: every fp32 operation is an explicitly rounded one (paired add.rn/mul.rn,
// __fadd_rn, __fmul_rn, __fdiv_rn), so no multiply-add is ever contracted into an FMA
// and each division is the IEEE one; integer<->float conversions use exact magic-number
// identities (below). The build also passes -fmad=false and keeps denormals (no -ftz).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

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

// 16 bytes global -> shared without passing through registers (both addresses 16-byte
// aligned), tracked by commit groups: cp_async_wait<N> returns once at most N of this
// thread's committed groups are still in flight.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------------
// Bulk copies into shared memory, tracked by an mbarrier (the transaction count of the
// barrier's current phase is raised by expect_tx and lowered as the bytes land).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned arrivals) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals)
               : "memory");
}
// Makes initialised barriers visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// One arrival that also expects `bytes` more bytes in the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// True once the phase with parity `parity` has completed (non-blocking test with the
// hardware's short built-in suspend).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// The wait after the first failed test, bounded by `limit_ns` of wall-clock time: false
// if the phase did not complete in time. Kept out of line so the common path (the phase
// has already completed) costs one test.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                               unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}
// bytes (a multiple of 16, both addresses 16-byte aligned) global -> shared; completion
// lowers the transaction count of `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, unsigned bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// 4 bytes global -> shared (asynchronous), and an arrival on `bar` once all of this
// thread's earlier cp.async copies have landed (counted in the barrier's arrivals).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
// Barrier among `nthreads` threads (a multiple of 32) of the CTA, by id (1..15; 0 is
// __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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

// 32 bytes as one 256-bit access (V8: the address is 32-byte aligned) or as two 128-bit
// accesses (the address is 16-byte aligned).
template <bool V8>
__device__ __forceinline__ U8x32 ld_vec32(const void* p) {
  if constexpr (V8) {
    return ld_stream_v8(p);
  } else {
    const uint4 a = ld_stream_v4(p), b = ld_stream_v4(static_cast<const uint8_t*>(p) + 16);
    U8x32 r;
    r.w[0] = a.x, r.w[1] = a.y, r.w[2] = a.z, r.w[3] = a.w;
    r.w[4] = b.x, r.w[5] = b.y, r.w[6] = b.z, r.w[7] = b.w;
    return r;
  }
}
template <bool V8>
__device__ __forceinline__ void st_vec32(void* p, const U8x32& v) {
  if constexpr (V8) {
    st_v8(p, v);
  } else {
    st_v4(p, make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]));
    st_v4(static_cast<uint8_t*>(p) + 16, make_uint4(v.w[4], v.w[5], v.w[6], v.w[7]));
  }
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

// Signed code i of a packed word (sign-extended by arithmetic shifts).
__device__ __forceinline__ int code_int8(uint32_t w, int i) {
  return static_cast<int>(w << (24 - 8 * i)) >> 24;
}
__device__ __forceinline__ int code_int4(uint32_t w, int i) {
  return static_cast<int>(w << (28 - 4 * i)) >> 28;
}

// ---------------------------------------------------------------------------------
// Paired fp32 arithmetic (sm_100 and later): one instruction applies the same IEEE
// single-precision operation to two independent lanes, each rounded to nearest even
// (no flush to zero). A product that feeds a sum is always written as the explicit
// fused form f2_fma (one rounding): the assembler may fuse a paired multiply followed
// by a paired add even when both carry .rn, so the two-step form is never relied on.
// ---------------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// a * b + c per lane, computed exactly and rounded once.
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// As f2_fma, rounded toward zero.
__device__ __forceinline__ f32x2 f2_fma_rz(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ---------------------------------------------------------------------------------
// Exact integer <-> float conversions without the conversion unit.
//
// Float -> code: for a real t with |t| < 2^22, fl(t + 1.5*2^23) lies in [2^23, 2^24),
// where the fp32 spacing is 1, so rounding the sum rounds t to the nearest integer with
// ties to even (1.5*2^23 is even); the bit pattern is 0x4B400000 + rint(t), whose low
// byte is rint(t) in two's complement. With t = x * inv formed inside one fused
// multiply-add, this is rint of the exact product.
// ---------------------------------------------------------------------------------
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// Code -> float: a code q offset to an unsigned u = q + 2^(bits-1) is byte-permuted into
// the low mantissa bits of 2^23, giving exactly 2^23 + u; subtracting 2^23 + 2^(bits-1)
// (exact: both operands are integers below 2^24) leaves exactly (float)q. (Measured on
// GB300 against shift + int-to-float conversion and against fp16-mantissa variants with
// mixed-precision adds, this is the highest-throughput form.)
__device__ __forceinline__ float byte_to_magic(uint32_t w, int j) {  // bits 0x4B0000bb
  return __uint_as_float(__byte_perm(w, 0x4B00u, 0x5440u + j));
}

// Eight INT4 codes (element i in nibble i) -> four pairs (2j, 2j+1) of exact floats.
__device__ __forceinline__ void int4x8_to_f2(uint32_t w, f32x2 q[4]) {
  const uint32_t lo = (w ^ 0x88888888u) & 0x0F0F0F0Fu;         // codes 0,2,4,6 (+8)
  const uint32_t hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;  // codes 1,3,5,7 (+8)
  const f32x2 off = f2(-8388616.0f, -8388616.0f);               // -(2^23 + 8)
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = f2_add(f2(byte_to_magic(lo, j), byte_to_magic(hi, j)), off);
}

// Eight INT4 codes -> exact floats, with the work split between the integer pipe and the
// fp32 pipe: one byte permute per byte (two codes) instead of one per code. With
// u = w ^ 0x88888888, byte j of u holds b = (q_2j + 8) + 16 (q_2j+1 + 8), and the permute
// gives the float B = 2^23 + b. Then, every step exact:
//   h      = rz(B / 16 + (1.5*2^23 - 2^19)) = 1.5*2^23 + (q_2j+1 + 8)  (rz drops (b%16)/16)
//   q_2j+1 = h - (1.5*2^23 + 8)
//   q_2j   = (B - (2^23 + 136)) - 16 q_2j+1
// ev[m] = (q_4m, q_4m+2), od[m] = (q_4m+1, q_4m+3), m = 0, 1.
__device__ __forceinline__ void int4x8_to_f2_eo(uint32_t w, f32x2 ev[2], f32x2 od[2]) {
  const uint32_t u = w ^ 0x88888888u;
  const f32x2 sixteenth = f2(0.0625f, 0.0625f), hi_base = f2(12058624.0f, 12058624.0f);
  const f32x2 hi_off = f2(-12582920.0f, -12582920.0f);  // -(1.5*2^23 + 8)
  const f32x2 b_off = f2(-8388744.0f, -8388744.0f);     // -(2^23 + 136)
  const f32x2 m16 = f2(-16.0f, -16.0f);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const f32x2 b = f2(byte_to_magic(u, 2 * m), byte_to_magic(u, 2 * m + 1));
    od[m] = f2_add(f2_fma_rz(b, sixteenth, hi_base), hi_off);
    ev[m] = f2_fma(od[m], m16, f2_add(b, b_off));
  }
}

// Four INT8 codes (element i in byte i) -> two pairs (0,1), (2,3) of exact floats.
__device__ __forceinline__ void int8x4_to_f2(uint32_t w, f32x2 q[2]) {
  const uint32_t u = w ^ 0x80808080u;              // q + 128 in every byte
  const f32x2 off = f2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  q[0] = f2_add(f2(byte_to_magic(u, 0), byte_to_magic(u, 1)), off);
  q[1] = f2_add(f2(byte_to_magic(u, 2), byte_to_magic(u, 3)), off);
}

// Low bytes of four rounded magic floats (as bits) -> one word [q0, q1, q2, q3].
__device__ __forceinline__ uint32_t gather_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// Eight rounded magic floats (pairs (0,1),(2,3),(4,5),(6,7)) -> one INT4 word.
__device__ __forceinline__ uint32_t pack_int4x8(const f32x2 r[4]) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) f2_split(r[j], v[2 * j], v[2 * j + 1]);
  const uint32_t ev = gather_low_bytes(__float_as_uint(v[0]), __float_as_uint(v[2]),
                                       __float_as_uint(v[4]), __float_as_uint(v[6]));
  const uint32_t od = gather_low_bytes(__float_as_uint(v[1]), __float_as_uint(v[3]),
                                       __float_as_uint(v[5]), __float_as_uint(v[7]));
  return (ev & 0x0F0F0F0Fu) | ((od << 4) & 0xF0F0F0F0u);
}

// Eight rounded magic floats in the layout of int4x8_to_f2_eo (pairs (0,2), (4,6),
// (1,3), (5,7)) -> one INT4 word.
__device__ __forceinline__ uint32_t pack_int4x8_eo(const f32x2 r[4]) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) f2_split(r[j], v[2 * j], v[2 * j + 1]);
  const uint32_t ev = gather_low_bytes(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                       __float_as_uint(v[2]), __float_as_uint(v[3]));
  const uint32_t od = gather_low_bytes(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                       __float_as_uint(v[6]), __float_as_uint(v[7]));
  return (ev & 0x0F0F0F0Fu) | ((od << 4) & 0xF0F0F0F0u);
}

// Four rounded magic floats (pairs (0,1),(2,3)) -> one INT8 word.
__device__ __forceinline__ uint32_t pack_int8x4(const f32x2 r[2]) {
  float v[4];
  f2_split(r[0], v[0], v[1]);
  f2_split(r[1], v[2], v[3]);
  return gather_low_bytes(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
}

// Codes of a pair: rint(x * inv) of the exact product, as magic floats. No clamp is
// needed: whenever inv is finite, |x| <= amax and inv <= (qmax / amax)(1 + 2^-24), so
// |x * inv| <= qmax (1 + 2^-24), which rounds to at most qmax.
__device__ __forceinline__ f32x2 round_codes(f32x2 x, f32x2 inv2) {
  return f2_fma(x, inv2, f2(kRoundMagic, kRoundMagic));
}

// Output element types of the dequantising kernels.
struct OutF16 {};
struct OutBF16 {};
struct OutF32 {};

// 16 consecutive fp32 values -> y[e .. e+16) of type OT (fp32: 64 bytes; fp16 / bf16:
// round to nearest even, 32 bytes), as 256-bit stores when y + e is 32-byte aligned (V8),
// else as 128-bit stores.
template <typename OT, bool V8>
__device__ __forceinline__ void store16(void* y, int64_t e, const float v[16]) {
  if constexpr (std::is_same_v<OT, OutF32>) {
    U8x32 a, b;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a.w[i] = __float_as_uint(v[i]);
      b.w[i] = __float_as_uint(v[8 + i]);
    }
    float* p = static_cast<float*>(y) + e;
    st_vec32<V8>(p, a);
    st_vec32<V8>(p + 8, b);
  } else {
    using TT = std::conditional_t<std::is_same_v<OT, OutF16>, F16, BF16>;
    U8x32 a;
#pragma unroll
    for (int i = 0; i < 8; ++i) a.w[i] = pack2(v[2 * i], v[2 * i + 1], TT());
    st_vec32<V8>(static_cast<uint16_t*>(y) + e, a);
  }
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
