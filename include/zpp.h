/*
 * zpp.h -- C ABI of the GB300 (sm_103a) ZeRO++ block-quantisation hot path.
 *
 * Pages cited (by title; the section follows the label):
 *   [ZeRO++ summary]  "ZeRO++: Extremely Efficient Collective Communication for Large
 *                      Model Training" (atlas.scime.ai summary)
 *   [ZeRO++ abstract] "ZeRO++: Extremely Efficient Collective Communication for Giant
 *                      Model Training" (mlsanity.com record, arXiv abstract)
 *   [LIT-102]         "LIT-102: ZeRO++: Extremely Efficient Collective Communication
 *                      for Giant Model Training" (anthology-of-the-sota record)
 *
 * What the calls compute (the pages fix the structure, not the formula; this is the
 * reading every entry point implements, bit for bit):
 *   per block of `block` consecutive elements (the last block may be shorter):
 *     amax  = max |x|;  scale = fp32(amax / qmax);  inv = fp32(qmax / amax)
 *     q     = clamp(rint_to_even(x * inv), -qmax, qmax),  qmax = 2^(bits-1) - 1,
 *             the product x * inv taken exactly (rounded once, to an integer)
 *     amax == 0 or inv not finite  ->  scale = 0 and every q = 0
 *   dequantise: y = fp32((float)q * scale), then round-to-nearest-even into y's type.
 *   reduce (the qgZ hops): sum = fma(q, scale, sum) per received chunk -- one rounding
 *   per term -- starting from +0.0f, sources in ascending order.
 *
 * Storage: INT8 codes are two's-complement bytes; INT4 codes are two's-complement
 * nibbles, element 2i in the LOW nibble of byte i and 2i+1 in the high nibble (an odd
 * trailing element leaves the high nibble 0). Scales are a separate fp32 array, one
 * per block, in block order.
 *
 * Virtual topology (qgZ): N nodes x M GPUs per node, W = N*M ranks, rank r = n*M + l.
 * Ranks are HBM buffers laid out back to back ([W][...]); the all-to-all exchanges are
 * index maps over them, no data is moved between the steps.
 *   E = elements per rank, S = E / W (the slice each rank owns), C = N*S (hop-1 chunk).
 *
 * Conventions for every entry point:
 *   - All buffer pointers are DEVICE pointers owned by the caller. The library
 *     allocates nothing, never synchronises, and only enqueues kernels on `stream`
 *     (0 = the legacy default stream).
 *   - Inputs and outputs must not overlap.
 *   - Arguments are checked on the host before any launch; on an error nothing is
 *     launched and nothing is written.
 *   - Alignment: element and code buffers (x, y, grads, codes, out, and the tensors of
 *     zpp_qgz_reorder_quant_tensors) must be 16-byte aligned; scale arrays 4-byte
 *     aligned. Element buffers that are also 32-byte aligned take 256-bit vector accesses,
 *     16-byte aligned ones 128-bit accesses; the results are the same bits.
 *   - n == 0 (or a zero-sized topology payload) returns ZPP_OK and launches nothing.
 *   - A launch failure is reported as ZPP_ERR_CUDA (from cudaGetLastError); an
 *     asynchronous fault surfaces at the caller's next synchronisation.
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef ZPP_H
#define ZPP_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define ZPP_API __attribute__((visibility("default")))
#else
#define ZPP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zpp_status {
  ZPP_OK = 0,
  ZPP_ERR_INVALID_ARG = 1, /* bad bits / block / size / topology / null pointer */
  ZPP_ERR_MISALIGNED = 2,  /* a pointer breaks the alignment rule above */
  ZPP_ERR_UNSUPPORTED = 3, /* a valid but unimplemented dtype combination */
  ZPP_ERR_CUDA = 4         /* the CUDA runtime reported an error at launch */
} zpp_status;

typedef enum zpp_dtype { ZPP_F16 = 0, ZPP_BF16 = 1, ZPP_F32 = 2 } zpp_dtype;

typedef struct zpp_topology {
  int32_t num_nodes;     /* N >= 1 */
  int32_t gpus_per_node; /* M >= 1 */
} zpp_topology;

/* A range [begin, end) of local GPU indices l (0 <= begin <= end <= M). The qgZ exchange
 * splits exactly by l: hop-1 chunk l of every rank feeds only the receivers with local
 * index l, whose hop-1 outputs feed only the hop-2 receivers with local index l. So the
 * three qgZ steps restricted to one range form an independent sub-pipeline, and the
 * ranges of a partition of [0, M) may run on different streams (the pipelining of the
 * intra- and inter-node hops, on one GPU). */
typedef struct zpp_local_range {
  int32_t begin;
  int32_t end;
} zpp_local_range;

/* Limits checked by every entry point. */
#define ZPP_MIN_BLOCK 64
#define ZPP_MAX_BLOCK 4096
#define ZPP_MAX_ELEMS (((int64_t)1) << 38)
#define ZPP_MAX_TENSORS 1024 /* tensors per bucket in zpp_qgz_reorder_quant_tensors */

/*
 * qwZ step 1 -- block-wise symmetric quantisation of a weight shard before the forward
 * all-gather ([ZeRO++ summary] Approach: block-wise INT8 weight quantisation;
 * [ZeRO++ abstract]: block-quantisation based all-gather; [LIT-102] Key takeaways:
 * block-wise rather than per-tensor). Also the INT4 gradient quantiser of qgZ.
 *   x      : [n] elements of x_dt (ZPP_F16 or ZPP_BF16; ZPP_F32 -> ZPP_ERR_UNSUPPORTED)
 *   n      : element count, 0 <= n <= ZPP_MAX_ELEMS
 *   block  : power of two in [64, 4096]
 *   bits   : 8 or 4
 *   codes  : out, zpp_code_bytes(n, bits) bytes
 *   scales : out, zpp_num_scales(n, block) floats
 * Shards whose sizes are multiples of `block` can be quantised in one call over their
 * concatenation: the result is identical to one call per shard.
 */
ZPP_API zpp_status zpp_quant_blockwise(const void* x, zpp_dtype x_dt, int64_t n, int32_t block,
                               int32_t bits, void* codes, float* scales, cudaStream_t stream);

/*
 * qwZ step 2 -- dequantisation of the gathered codes after the all-gather
 * ([ZeRO++ summary] Approach; [ZeRO++ abstract]: block-quantisation based all-gather).
 *   codes  : [zpp_code_bytes(n, bits)] bytes; scales: [zpp_num_scales(n, block)] floats
 *   y      : out, [n] elements of y_dt (ZPP_F16, ZPP_BF16 or ZPP_F32)
 * Other arguments as in zpp_quant_blockwise.
 */
ZPP_API zpp_status zpp_dequant_blockwise(const void* codes, const float* scales, int64_t n,
                                 int32_t block, int32_t bits, void* y, zpp_dtype y_dt,
                                 cudaStream_t stream);

/*
 * qgZ step 1 -- tensor-slice reordering plus block quantisation of every rank's
 * gradient before the 2-hop all-to-all ([ZeRO++ summary] Approach: slices reordered
 * so each reduced slice lands on its owner; INT4 gradient reduction).
 * Each rank's E elements are W slices of S; original slice j = n_d*M + l_d (owned by
 * rank j) is written at position p = l_d*N + n_d, so the reordered buffer is M chunks
 * of C = N*S, chunk l going to local peer l in hop 1. Quantisation then runs over the
 * reordered buffer (blocks never straddle slices).
 *   grads          : [W][E] elements of g_dt (ZPP_F16 or ZPP_BF16)
 *   elems_per_rank : E, a multiple of W*block, E < 2^31
 *   bits           : 4 (the pages' INT4); 8 is accepted as an extension
 *   codes          : out, [W][zpp_code_bytes(E, bits)]
 *   scales         : out, [W][E/block]
 */
ZPP_API zpp_status zpp_qgz_reorder_quant(const void* grads, zpp_dtype g_dt, int64_t elems_per_rank,
                                 int32_t block, int32_t bits, zpp_topology topo,
                                 void* codes, float* scales, cudaStream_t stream);

/*
 * qgZ step 1 with the bucket flatten fused in. A rank's gradient bucket is usually the
 * concatenation of many parameter gradients; this call reads them where they are
 * instead of from a flattened copy, and writes exactly (bit for bit) what
 * zpp_qgz_reorder_quant writes for the bucket whose rank r holds, in order, its copies of
 * tensors 0..num_tensors-1 ([ZeRO++ summary] Approach: slices reordered for correct
 * placement). The flattening copy -- a full read and write of the bucket -- is saved.
 *   tensors     : HOST array [num_tensors] of device pointers; tensor t holds the W ranks'
 *                 copies back to back ([W][sizes[t]] elements of g_dt), 16-byte aligned
 *   sizes       : HOST array [num_tensors], elements per rank of tensor t: a multiple of
 *                 16 (else ZPP_ERR_MISALIGNED), 0 allowed (its pointer is then not read)
 *   num_tensors : 1 .. ZPP_MAX_TENSORS
 * E = the sum of sizes must satisfy the rules of zpp_qgz_reorder_quant (a multiple of
 * W*block, E < 2^31); codes and scales are as there. Tensors of one rank may cross slice
 * and block boundaries freely. Both host arrays are read during the call only.
 */
ZPP_API zpp_status zpp_qgz_reorder_quant_tensors(const void* const* tensors, const int64_t* sizes,
                                                 int32_t num_tensors, zpp_dtype g_dt,
                                                 int32_t block, int32_t bits, zpp_topology topo,
                                                 void* codes, float* scales, cudaStream_t stream);

/*
 * qgZ step 2 -- the fused kernel of the intra-node hop: every receiver (n, l)
 * dequantises chunk l of the M ranks of its node, sums them in fp32 (l' ascending) and
 * requantises the sums by blocks for the inter-node hop ([ZeRO++ summary] Approach:
 * dequantise before reduction; Measured effects table: fusion kernel; [LIT-102] Key
 * takeaways: reduce locally in higher precision). K = M chunks are read once.
 *   codes, scales  : the outputs of zpp_qgz_reorder_quant
 *   out_codes      : out, [W][zpp_code_bytes(C, bits)]
 *   out_scales     : out, [W][C/block]
 */
ZPP_API zpp_status zpp_dequant_reduce_requant(const void* codes, const float* scales,
                                      int64_t elems_per_rank, int32_t block, int32_t bits,
                                      zpp_topology topo, void* out_codes, float* out_scales,
                                      cudaStream_t stream);

/*
 * qgZ step 3 -- the inter-node hop's final dequantise-reduce: receiver (n, l)
 * dequantises slice n of the hop-1 output of rank (n', l) for n' = 0..N-1 and sums in
 * fp32 (n' ascending). The result is the SUM over all W ranks of the receiver's own
 * slice; scaling by 1/W for an average is left to the caller ([ZeRO++ summary]
 * Approach; [ZeRO++ abstract]: quantised gradient averaging).
 *   codes, scales  : the outputs of zpp_dequant_reduce_requant
 *   out            : out, [W][S] fp32
 */
ZPP_API zpp_status zpp_dequant_reduce(const void* codes, const float* scales, int64_t elems_per_rank,
                              int32_t block, int32_t bits, zpp_topology topo, float* out,
                              cudaStream_t stream);

/*
 * qgZ step 3 with the average folded in ([ZeRO++ abstract]: the gradient step averages
 * the ranks' gradients). Computes the same sums as zpp_dequant_reduce, multiplies each by
 * post_scale (one fp32 rounding; pass 1/W for the average, exact when W is a power of
 * two) and stores the result as out_dt with round-to-nearest-even.
 *   post_scale : finite, else ZPP_ERR_INVALID_ARG
 *   out        : out, [W][S] elements of out_dt (ZPP_F16, ZPP_BF16 or ZPP_F32)
 * Other arguments as in zpp_dequant_reduce.
 */
ZPP_API zpp_status zpp_dequant_reduce_scaled(const void* codes, const float* scales,
                                             int64_t elems_per_rank, int32_t block, int32_t bits,
                                             zpp_topology topo, float post_scale, void* out,
                                             zpp_dtype out_dt, cudaStream_t stream);

/*
 * The three qgZ steps restricted to the local indices of `range` ([ZeRO++ summary]
 * Approach: overlapped intra- and inter-node pipelining). Buffers have the full layouts
 * of the unrestricted calls; only the parts that belong to the range are read or written:
 *   zpp_qgz_reorder_quant_range     writes chunks l in range of every rank's codes/scales
 *   zpp_dequant_reduce_requant_range writes the hop-1 output of receivers (n, l), l in range
 *   zpp_dequant_reduce_scaled_range  writes the owner slices of ranks (n, l), l in range
 * An empty range returns ZPP_OK and launches nothing; a range outside [0, M] is
 * ZPP_ERR_INVALID_ARG. Results are bit-identical to the unrestricted calls.
 */
ZPP_API zpp_status zpp_qgz_reorder_quant_range(const void* grads, zpp_dtype g_dt,
                                               int64_t elems_per_rank, int32_t block,
                                               int32_t bits, zpp_topology topo,
                                               zpp_local_range range, void* codes,
                                               float* scales, cudaStream_t stream);
ZPP_API zpp_status zpp_dequant_reduce_requant_range(const void* codes, const float* scales,
                                                    int64_t elems_per_rank, int32_t block,
                                                    int32_t bits, zpp_topology topo,
                                                    zpp_local_range range, void* out_codes,
                                                    float* out_scales, cudaStream_t stream);
ZPP_API zpp_status zpp_dequant_reduce_scaled_range(const void* codes, const float* scales,
                                                   int64_t elems_per_rank, int32_t block,
                                                   int32_t bits, zpp_topology topo,
                                                   zpp_local_range range, float post_scale,
                                                   void* out, zpp_dtype out_dt,
                                                   cudaStream_t stream);

/*
 * The three qgZ steps as one real rank runs them, on its own buffers, with the two
 * all-to-all exchanges between them left to the caller's collectives ([ZeRO++ summary]
 * Approach: 2-hop all-to-all; the virtual-layout calls above run the same kernels with the
 * exchanges as index maps). For rank r = n*M + l of topology {N, M}, W = N*M, S = E/W,
 * C = N*S:
 *
 * zpp_qgz_reorder_quant_local -- step 1 on this rank's E gradient elements: exactly row r
 *   of what zpp_qgz_reorder_quant writes (the reorder does not depend on r). Chunk l' (C
 *   elements at offset l'*C) of the result is what goes to local peer l' in hop 1; only
 *   the chunks l' in `range` are written ({0, M}: all), so each can be produced just before
 *   its send.
 *   grads : [E] elements of g_dt; codes: out, [zpp_code_bytes(E, bits)]; scales: out, [E/block]
 *   Rules as for zpp_qgz_reorder_quant_range.
 *
 * zpp_dequant_reduce_requant_local -- the fused intra-node hop on the chunks this rank
 *   received: chunk l of each of its node's M ranks, in local-index order, `sources` = M
 *   chunks of `chunk` = C elements back to back. Writes exactly row r of what
 *   zpp_dequant_reduce_requant writes.
 *   codes : [sources][zpp_code_bytes(chunk, bits)]; scales: [sources][chunk/block]
 *   out_codes : out, [zpp_code_bytes(chunk, bits)]; out_scales: out, [chunk/block]
 *
 * zpp_dequant_reduce_local -- the final inter-node hop on the slices this rank received:
 *   slice n of the hop-1 output of ranks (n', l), n' = 0..N-1 ascending, `sources` = N
 *   slices of `slice` = S elements back to back. Writes exactly row r of what
 *   zpp_dequant_reduce_scaled writes (post_scale 1 and fp32 out: zpp_dequant_reduce).
 *   codes : [sources][zpp_code_bytes(slice, bits)]; scales: [sources][slice/block]
 *   out   : out, [slice] elements of out_dt; post_scale: finite
 *
 * For the last two: block a power of two in [64, 4096], bits 4 or 8, 1 <= sources <= 65535,
 * chunk (slice) a multiple of block below 2^31 (0: ZPP_OK, nothing launched), else
 * ZPP_ERR_INVALID_ARG. Alignment and ownership as for every call.
 */
ZPP_API zpp_status zpp_qgz_reorder_quant_local(const void* grads, zpp_dtype g_dt,
                                               int64_t elems_per_rank, int32_t block, int32_t bits,
                                               zpp_topology topo, zpp_local_range range,
                                               void* codes, float* scales, cudaStream_t stream);
ZPP_API zpp_status zpp_dequant_reduce_requant_local(const void* codes, const float* scales,
                                                    int64_t chunk, int32_t block, int32_t bits,
                                                    int32_t sources, void* out_codes,
                                                    float* out_scales, cudaStream_t stream);
ZPP_API zpp_status zpp_dequant_reduce_local(const void* codes, const float* scales, int64_t slice,
                                            int32_t block, int32_t bits, int32_t sources,
                                            float post_scale, void* out, zpp_dtype out_dt,
                                            cudaStream_t stream);

/* Bytes of packed codes for n elements: n for INT8, ceil(n/2) for INT4; -1 on bad bits. */
ZPP_API int64_t zpp_code_bytes(int64_t n, int32_t bits);

/* Number of scales for n elements: ceil(n / block); -1 on a bad block. */
ZPP_API int64_t zpp_num_scales(int64_t n, int32_t block);

/* Static, never-NULL description of a status code. */
ZPP_API const char* zpp_status_string(zpp_status status);

/*
 * Fault word of the current device (no counterpart in the pages). Kernels that wait for
 * data in flight (the INT8 fused-hop kernel waits on shared-memory barriers completed by
 * bulk copies) bound every wait to about a second; a wait that runs out sets a bit here,
 * the kernel still ends, and its outputs are unspecified. Bits: 1 and 2 -- a wait of the
 * INT8 fused hop ran out; 4 -- zpp_wait_selftest ran out (as it always does).
 *   flags : out, the word (0 when nothing ran out since the last clear)
 *   clear : nonzero -> zero the word after reading it
 * Unlike the other calls this one synchronises with the device (it copies the word back);
 * call it after the work it should cover has been synchronised.
 */
ZPP_API zpp_status zpp_device_fault(uint32_t* flags, int32_t clear);

/*
 * Diagnostic (no counterpart in the pages): launches one warp that waits on a
 * shared-memory barrier nothing completes, bounded by limit_ns nanoseconds (1 ns .. 10 s,
 * else ZPP_ERR_INVALID_ARG), then sets bit 4 of the fault word and ends. It exercises the
 * bounded wait and the fault report on the device without a fault of any kind.
 */
ZPP_API zpp_status zpp_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

/*
 * Measurement helper (no counterpart in the pages): a 256-bit streaming device copy
 * used as the same-run HBM reference next to the kernels above.
 *   src, dst : 32-byte aligned device buffers; bytes: a multiple of 32.
 */
ZPP_API zpp_status zpp_device_copy(const void* src, void* dst, int64_t bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ZPP_H */
