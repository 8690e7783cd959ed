/*
 * zpp_oracle.c -- plain, slow, scalar CPU oracle for the ZeRO++ block-quantisation
 * hot path (qwZ and qgZ).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
 * file. Its only users are the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark. It shares no code, header, table or constant with the CUDA
 * library: every conversion and every index map below is written here again.
 *
 * Pages cited (by title; sections named after the label):
 *   [ZeRO++ summary]  "ZeRO++: Extremely Efficient Collective Communication for Large
 *                      Model Training" (atlas.scime.ai AI-written summary)
 *   [ZeRO++ abstract] "ZeRO++: Extremely Efficient Collective Communication for Giant
 *                      Model Training" (mlsanity.com record, "Abstract (arXiv)")
 *   [LIT-102]         "LIT-102: ZeRO++: Extremely Efficient Collective Communication
 *                      for Giant Model Training" (anthology-of-the-sota record)
 *
 * The pages fix the structure of the method (block-wise INT8 weights, INT4 gradients,
 * slice reordering, dequantise before a higher-precision reduction, two hops) but no
 * formula. The arithmetic below is the plainest reading consistent with them:
 *
 *   x      = (float) input                         (exact for fp16 / bf16)
 *   amax   = max |x| over the block
 *   qmax   = 2^(bits-1) - 1                        (127 for INT8, 7 for INT4: symmetric)
 *   scale  = amax / qmax,  inv = qmax / amax       (two IEEE fp32 divisions per block)
 *   q      = clamp(rint(x * inv), -qmax, qmax)     (rint: ties to even, applied to the
 *                                                   exact product x * inv)
 *   if amax == 0 or inv is not finite: scale = 0, q = 0 for the whole block
 *   y      = (float) q * scale                     (then RNE cast to the output type)
 *   sum    = fma(q, scale, sum) per received chunk (one rounding per term; sums start at
 *                                                   +0.0f, sources in ascending order)
 *
 * The products x * inv are formed exactly in double (24-bit by 24-bit significands fit in
 * 53 bits) and rounded to an integer once; the hop sums add each dequantised term with a
 * single rounding (C99 fmaf). Nothing else is fused: the file is compiled with
 * -ffp-contract=off and without fast-math. INT4 codes are two's-complement nibbles, element 2i in the low
 * nibble of byte i, element 2i+1 in the high nibble; a trailing odd element leaves the
 * high nibble 0. Scales are a separate fp32 array, one per block.
 *
 * Parallelism: OpenMP over independent blocks / receivers only (results do not depend
 * on the thread count).
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2 };

/* ---------------------------------------------------------------------------------
 * Threads used by the parallel loops (for the CPU-baseline timing).
 * ------------------------------------------------------------------------------- */
int or_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ---------------------------------------------------------------------------------
 * Floating-point storage formats, written from their IEEE-754 / bfloat16 definitions.
 * ------------------------------------------------------------------------------- */

/* binary16 -> binary32 (exact). value = (-1)^s * 2^(e-15) * 1.m, or 2^-14 * 0.m. */
float or_f16_to_f32(uint16_t h) {
  uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
  float mag;
  if (e == 0)
    mag = ldexpf((float)m, -24);
  else if (e == 31)
    mag = m ? NAN : INFINITY;
  else
    mag = ldexpf((float)(m | 0x400u), (int)e - 25);
  return s ? -mag : mag;
}

/* binary32 -> binary16, round to nearest even. The scaling by a power of two is exact
 * in double, and nearbyint() rounds ties to even under the default rounding mode. */
uint16_t or_f32_to_f16(float f) {
  uint16_t s = signbit(f) ? 0x8000u : 0u;
  if (isnan(f)) return (uint16_t)(s | 0x7e00u);
  double a = fabs((double)f);
  if (a >= 65520.0) return (uint16_t)(s | 0x7c00u); /* halfway to 2^16 and above: inf */
  if (a < ldexp(1.0, -14)) {                        /* subnormal: units of 2^-24 */
    double m = nearbyint(a * ldexp(1.0, 24));       /* 1024 encodes the least normal */
    return (uint16_t)(s | (uint16_t)m);
  }
  int e2;
  frexp(a, &e2);                                    /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;
  double m = nearbyint(a * ldexp(1.0, 10 - E));     /* in [1024, 2048] */
  if (m == 2048.0) {
    m = 1024.0;
    E += 1;
  }
  if (E > 15) return (uint16_t)(s | 0x7c00u);
  return (uint16_t)(s | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* bfloat16 is the upper half of a binary32. */
float or_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> bfloat16, round to nearest even on the dropped 16 bits. */
uint16_t or_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t hi = u >> 16, lo = u & 0xffffu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u; /* carry may reach inf */
  return (uint16_t)hi;
}

static float load_value(const void* x, int dtype, int64_t i) {
  if (dtype == OR_F16) return or_f16_to_f32(((const uint16_t*)x)[i]);
  if (dtype == OR_BF16) return or_bf16_to_f32(((const uint16_t*)x)[i]);
  return ((const float*)x)[i];
}

static void store_value(void* y, int dtype, int64_t i, float v) {
  if (dtype == OR_F16)
    ((uint16_t*)y)[i] = or_f32_to_f16(v);
  else if (dtype == OR_BF16)
    ((uint16_t*)y)[i] = or_f32_to_bf16(v);
  else
    ((float*)y)[i] = v;
}

/* ---------------------------------------------------------------------------------
 * Block quantisation of fp32 values ([ZeRO++ summary] Approach: block-wise INT8
 * weights and INT4 gradients; [LIT-102] Key takeaways: block-wise rather than
 * per-tensor scaling).
 * ------------------------------------------------------------------------------- */

/* One block of `len` values -> `len` signed codes and one fp32 scale. */
static void quant_block(const float* v, int64_t len, int bits, int8_t* q, float* scale_out) {
  const float qmax = (float)((1 << (bits - 1)) - 1);
  float amax = 0.0f;
  for (int64_t i = 0; i < len; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float scale = amax / qmax;
  float inv = qmax / amax;
  if (amax == 0.0f || !isfinite(inv)) {
    for (int64_t i = 0; i < len; ++i) q[i] = 0;
    *scale_out = 0.0f;
    return;
  }
  for (int64_t i = 0; i < len; ++i) {
    double t = nearbyint((double)v[i] * (double)inv); /* exact product, one rounding */
    if (t > qmax) t = qmax;
    if (t < -qmax) t = -qmax;
    q[i] = (int8_t)t;
  }
  *scale_out = scale;
}

/* Signed codes -> storage bytes: INT8 as two's-complement bytes; INT4 as nibbles with
 * element 2i low and 2i+1 high; an odd trailing element leaves the high nibble 0. */
static void pack_codes(const int8_t* q, int64_t n, int bits, uint8_t* out) {
  if (bits == 8) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)q[i];
    return;
  }
  for (int64_t i = 0; 2 * i < n; ++i) {
    uint8_t lo = (uint8_t)(q[2 * i] & 0xf);
    uint8_t hi = (2 * i + 1 < n) ? (uint8_t)(q[2 * i + 1] & 0xf) : 0u;
    out[i] = (uint8_t)(lo | (hi << 4));
  }
}

/* Storage bytes -> signed code of element i. */
static int code_at(const uint8_t* codes, int bits, int64_t i) {
  if (bits == 8) return (int)(int8_t)codes[i];
  int nib = (i & 1) ? (codes[i >> 1] >> 4) : (codes[i >> 1] & 0xf);
  return nib >= 8 ? nib - 16 : nib;
}

int64_t or_code_bytes(int64_t n, int bits) { return bits == 8 ? n : (n + 1) / 2; }

/* Quantise n fp32 values by blocks of `block` (the last block may be shorter). */
static int quant_f32(const float* v, int64_t n, int64_t block, int bits, uint8_t* codes,
                     float* scales) {
  int8_t* q = (int8_t*)malloc((size_t)(n > 0 ? n : 1));
  if (!q) return -1;
  int64_t nb = (n + block - 1) / block;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nb; ++b) {
    int64_t lo = b * block, len = (n - lo < block) ? n - lo : block;
    quant_block(v + lo, len, bits, q + lo, &scales[b]);
  }
  pack_codes(q, n, bits, codes);
  free(q);
  return 0;
}

/* qwZ quantise: input of `dtype` (fp16/bf16/fp32 bit patterns) -> codes + scales. */
int or_quant_blockwise(const void* x, int dtype, int64_t n, int64_t block, int bits,
                       uint8_t* codes, float* scales) {
  if (n <= 0) return 0;
  float* v = (float*)malloc((size_t)n * sizeof(float));
  if (!v) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) v[i] = load_value(x, dtype, i);
  int rc = quant_f32(v, n, block, bits, codes, scales);
  free(v);
  return rc;
}

/* qwZ dequantise: y = (float)q * scale, then cast to `y_dtype` with RNE. */
int or_dequant_blockwise(const uint8_t* codes, const float* scales, int64_t n, int64_t block,
                         int bits, void* y, int y_dtype) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)code_at(codes, bits, i) * scales[i / block];
    store_value(y, y_dtype, i, v);
  }
  return 0;
}

/* ---------------------------------------------------------------------------------
 * qgZ ([ZeRO++ summary] Approach: 2-hop all-to-all INT4 gradient reduction that
 * dequantises before reducing, with tensor slice reordering for correct placement;
 * [LIT-102] Key takeaways: one quantisation per exchange, local reduction in higher
 * precision).
 *
 * Topology: N nodes x M GPUs per node, W = N*M ranks, rank r = n*M + l. Each rank holds
 * E gradient elements, split into W slices of S = E/W; original slice j is the part
 * rank j will own after the reduction.
 * ------------------------------------------------------------------------------- */

/* Reordered position of original slice j = n_d*M + l_d: p = l_d*N + n_d. The reordered
 * buffer is then M chunks of N*S, chunk l_d going to local peer l_d in hop 1. */
int64_t or_reorder_position(int64_t j, int N, int M) {
  int64_t n_d = j / M, l_d = j % M;
  return l_d * N + n_d;
}

/* Hop 1 (intra-node all-to-all): receiver (n, l) takes chunk l of every rank of its node. */
static int64_t hop1_source(int n, int M, int lp) { return (int64_t)n * M + lp; }
/* Hop 2 (inter-node all-to-all): receiver (n, l) takes slice n of the hop-1 output of
 * rank (n', l) on every node n'. */
static int64_t hop2_source(int np, int M, int l) { return (int64_t)np * M + l; }

/* Reorder one rank's E fp32 values slice-wise (no arithmetic). */
void or_reorder_slices(const float* src, int64_t E, int N, int M, float* dst) {
  int64_t W = (int64_t)N * M, S = E / W;
  for (int64_t j = 0; j < W; ++j)
    memcpy(dst + or_reorder_position(j, N, M) * S, src + j * S, (size_t)S * sizeof(float));
}

/* Step a3: per source rank, reorder then quantise by blocks.
 * grads [W][E] of dtype -> codes [W][code_bytes(E)], scales [W][E/block]. */
int or_qgz_reorder_quant(const void* grads, int dtype, int64_t E, int64_t block, int bits,
                         int N, int M, uint8_t* codes, float* scales) {
  int64_t W = (int64_t)N * M;
  float* v = (float*)malloc((size_t)E * sizeof(float));
  float* p = (float*)malloc((size_t)E * sizeof(float));
  if (!v || !p) {
    free(v);
    free(p);
    return -1;
  }
  const size_t esz = dtype == OR_F32 ? 4 : 2;
  for (int64_t r = 0; r < W; ++r) {
    const char* row = (const char*)grads + (size_t)(r * E) * esz;
    for (int64_t i = 0; i < E; ++i) v[i] = load_value(row, dtype, i);
    or_reorder_slices(v, E, N, M, p);
    if (quant_f32(p, E, block, bits, codes + r * or_code_bytes(E, bits), scales + r * (E / block))) {
      free(v);
      free(p);
      return -1;
    }
  }
  free(v);
  free(p);
  return 0;
}

/* Step a5 (hop 1 + the fused kernel of the pages): receiver (n, l) dequantises chunk l
 * of each rank (n, l'), sums in fp32 over l' = 0..M-1 ascending from +0.0f (each term
 * q * scale added with one rounding), then requantises the N*S sums by blocks.
 * codes/scales: the output of step a3. out_codes [W][code_bytes(N*S)], out_scales
 * [W][N*S/block]. */
int or_dequant_reduce_requant(const uint8_t* codes, const float* scales, int64_t E,
                              int64_t block, int bits, int N, int M, uint8_t* out_codes,
                              float* out_scales) {
  int64_t W = (int64_t)N * M, S = E / W, C = (int64_t)N * S;
  float* acc = (float*)malloc((size_t)C * sizeof(float));
  if (!acc) return -1;
  for (int n = 0; n < N; ++n) {
    for (int l = 0; l < M; ++l) {
      int64_t r = (int64_t)n * M + l;
#pragma omp parallel for schedule(static)
      for (int64_t e = 0; e < C; ++e) {
        float a = 0.0f;
        for (int lp = 0; lp < M; ++lp) {
          int64_t src = hop1_source(n, M, lp);
          int64_t idx = (int64_t)l * C + e; /* chunk l of the reordered source */
          a = fmaf((float)code_at(codes + src * or_code_bytes(E, bits), bits, idx),
                   scales[src * (E / block) + idx / block], a);
        }
        acc[e] = a;
      }
      if (quant_f32(acc, C, block, bits, out_codes + r * or_code_bytes(C, bits),
                    out_scales + r * (C / block))) {
        free(acc);
        return -1;
      }
    }
  }
  free(acc);
  return 0;
}

/* Step a7 (hop 2): receiver (n, l) dequantises slice n of the hop-1 output of every rank
 * (n', l) and sums over n' = 0..N-1 ascending from +0.0f (one rounding per term).
 * out [W][S] fp32 (a sum; any averaging factor is left to the caller). */
int or_dequant_reduce(const uint8_t* codes1, const float* scales1, int64_t E, int64_t block,
                      int bits, int N, int M, float* out) {
  int64_t W = (int64_t)N * M, S = E / W, C = (int64_t)N * S;
  for (int n = 0; n < N; ++n) {
    for (int l = 0; l < M; ++l) {
      int64_t r = (int64_t)n * M + l;
#pragma omp parallel for schedule(static)
      for (int64_t e = 0; e < S; ++e) {
        float a = 0.0f;
        for (int np = 0; np < N; ++np) {
          int64_t src = hop2_source(np, M, l);
          int64_t idx = (int64_t)n * S + e; /* slice n of the hop-1 output */
          a = fmaf((float)code_at(codes1 + src * or_code_bytes(C, bits), bits, idx),
                   scales1[src * (C / block) + idx / block], a);
        }
        out[r * S + e] = a;
      }
    }
  }
  return 0;
}

/* Step a7 with the average folded in ([ZeRO++ abstract]: the gradient step averages):
 * the hop-2 sum of or_dequant_reduce multiplied by post_scale (one fp32 rounding; pass
 * 1/W for the average) and stored as out_dtype with round-to-nearest-even. */
int or_dequant_reduce_scaled(const uint8_t* codes1, const float* scales1, int64_t E,
                             int64_t block, int bits, int N, int M, float post_scale, void* out,
                             int out_dtype) {
  int64_t W = (int64_t)N * M, S = E / W;
  float* sum = (float*)malloc((size_t)(W * S) * sizeof(float));
  if (!sum) return -1;
  or_dequant_reduce(codes1, scales1, E, block, bits, N, M, sum);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < W * S; ++i) store_value(out, out_dtype, i, sum[i] * post_scale);
  free(sum);
  return 0;
}

/* One receiver's hops on the chunks it was sent, as a real rank runs them after each
 * all-to-all ([ZeRO++ summary] Approach: dequantise the received chunks, reduce in higher
 * precision; [LIT-102] Key takeaways). The K received chunks of `len` elements lie back to
 * back, sources in the order they are summed: codes [K][code_bytes(len)], scales
 * [K][len/block]. Each output element is acc = fma(q, scale, acc) over k = 0..K-1 from
 * +0.0f. */

/* Hop 1: the sums requantised by blocks -> out_codes [code_bytes(len)], out_scales. */
int or_dequant_reduce_requant_chunks(const uint8_t* codes, const float* scales, int64_t len,
                                     int64_t block, int bits, int K, uint8_t* out_codes,
                                     float* out_scales) {
  float* acc = (float*)malloc((size_t)(len > 0 ? len : 1) * sizeof(float));
  if (!acc) return -1;
  const int64_t cb = or_code_bytes(len, bits), nb = len / block;
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < len; ++e) {
    float a = 0.0f;
    for (int k = 0; k < K; ++k)
      a = fmaf((float)code_at(codes + k * cb, bits, e), scales[k * nb + e / block], a);
    acc[e] = a;
  }
  int rc = quant_f32(acc, len, block, bits, out_codes, out_scales);
  free(acc);
  return rc;
}

/* Hop 2: the sums times post_scale (one fp32 rounding), stored as out_dtype -> out [len]. */
int or_dequant_reduce_chunks(const uint8_t* codes, const float* scales, int64_t len,
                             int64_t block, int bits, int K, float post_scale, void* out,
                             int out_dtype) {
  const int64_t cb = or_code_bytes(len, bits), nb = len / block;
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < len; ++e) {
    float a = 0.0f;
    for (int k = 0; k < K; ++k)
      a = fmaf((float)code_at(codes + k * cb, bits, e), scales[k * nb + e / block], a);
    store_value(out, out_dtype, e, a * post_scale);
  }
  return 0;
}

/* The same two hops with quantisation switched off (fp32 pass-through), used to check
 * placement. reorder = 0 skips the slice reordering (the wrong layout). x [W][E] ->
 * out [W][S]. */
int or_qgz_passthrough(const float* x, int64_t E, int N, int M, int reorder, float* out) {
  int64_t W = (int64_t)N * M, S = E / W, C = (int64_t)N * S;
  float* sent = (float*)malloc((size_t)(W * E) * sizeof(float));
  float* hop1 = (float*)malloc((size_t)(W * C) * sizeof(float));
  if (!sent || !hop1) {
    free(sent);
    free(hop1);
    return -1;
  }
  for (int64_t r = 0; r < W; ++r) {
    if (reorder)
      or_reorder_slices(x + r * E, E, N, M, sent + r * E);
    else
      memcpy(sent + r * E, x + r * E, (size_t)E * sizeof(float));
  }
  for (int n = 0; n < N; ++n)
    for (int l = 0; l < M; ++l)
      for (int64_t e = 0; e < C; ++e) {
        float a = 0.0f;
        for (int lp = 0; lp < M; ++lp) a = a + sent[hop1_source(n, M, lp) * E + (int64_t)l * C + e];
        hop1[((int64_t)n * M + l) * C + e] = a;
      }
  for (int n = 0; n < N; ++n)
    for (int l = 0; l < M; ++l)
      for (int64_t e = 0; e < S; ++e) {
        float a = 0.0f;
        for (int np = 0; np < N; ++np) a = a + hop1[hop2_source(np, M, l) * C + (int64_t)n * S + e];
        out[((int64_t)n * M + l) * S + e] = a;
      }
  free(sent);
  free(hop1);
  return 0;
}

/* Rounding mode check for the Python side: the oracle assumes round-to-nearest. */
int or_rounding_is_nearest(void) { return fegetround() == FE_TONEAREST; }
