// zpp_abi.cu -- the extern "C" boundary of libzpp: argument checks (before any launch),
// kernel selection, status codes, and the same-run 256-bit copy kernel.
#include <zpp.h>

#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {

// K6: streaming copy. Each CTA copies 4 x 256 consecutive 32-byte vectors (all loads
// in flight before the stores) and exits.
__global__ void __launch_bounds__(kThreads) k_copy(const U8x32* __restrict__ src,
                                                   U8x32* __restrict__ dst, int64_t nvec) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads * 4 + threadIdx.x;
  U8x32 r[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (base + u * kThreads < nvec) r[u] = ld_stream_v8(src + base + u * kThreads);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (base + u * kThreads < nvec) st_v8(dst + base + u * kThreads, r[u]);
}

cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, cudaStream_t s) {
  const int64_t nvec = bytes / 32;
  const int grid = tile_grid(nvec, kThreads * 4);
  k_copy<<<grid, kThreads, 0, s>>>(static_cast<const U8x32*>(src), static_cast<U8x32*>(dst), nvec);
  return cudaGetLastError();
}

}  // namespace zpp

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_block(int32_t block) {
  return block >= ZPP_MIN_BLOCK && block <= ZPP_MAX_BLOCK && (block & (block - 1)) == 0;
}

bool valid_bits(int32_t bits) { return bits == 4 || bits == 8; }

zpp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ZPP_OK : ZPP_ERR_CUDA; }

// Shared checks of the three qgZ entry points; on success W is set.
zpp_status check_topology(int64_t E, int32_t block, int32_t bits, zpp_topology t, int64_t* W) {
  if (!valid_bits(bits) || !valid_block(block)) return ZPP_ERR_INVALID_ARG;
  if (t.num_nodes < 1 || t.gpus_per_node < 1) return ZPP_ERR_INVALID_ARG;
  const int64_t w = static_cast<int64_t>(t.num_nodes) * t.gpus_per_node;
  if (w > 65535) return ZPP_ERR_INVALID_ARG;  // ranks index grid dimensions
  if (E < 0 || E >= (int64_t{1} << 31)) return ZPP_ERR_INVALID_ARG;
  if (E % (w * block) != 0) return ZPP_ERR_INVALID_ARG;
  if (w * E > ZPP_MAX_ELEMS) return ZPP_ERR_INVALID_ARG;
  *W = w;
  return ZPP_OK;
}

bool valid_range(zpp_local_range r, zpp_topology t) {
  return r.begin >= 0 && r.begin <= r.end && r.end <= t.gpus_per_node;
}

zpp_local_range full_range(zpp_topology t) { return zpp_local_range{0, t.gpus_per_node}; }

}  // namespace

extern "C" {

int64_t zpp_code_bytes(int64_t n, int32_t bits) {
  if (n < 0 || !valid_bits(bits)) return -1;
  return bits == 8 ? n : (n + 1) / 2;
}

int64_t zpp_num_scales(int64_t n, int32_t block) {
  if (n < 0 || block <= 0) return -1;
  return (n + block - 1) / block;
}

const char* zpp_status_string(zpp_status s) {
  switch (s) {
    case ZPP_OK: return "ZPP_OK";
    case ZPP_ERR_INVALID_ARG: return "ZPP_ERR_INVALID_ARG: invalid argument";
    case ZPP_ERR_MISALIGNED: return "ZPP_ERR_MISALIGNED: pointer alignment rule broken";
    case ZPP_ERR_UNSUPPORTED: return "ZPP_ERR_UNSUPPORTED: unsupported dtype combination";
    case ZPP_ERR_CUDA: return "ZPP_ERR_CUDA: CUDA runtime error at launch";
  }
  return "unknown zpp_status";
}

zpp_status zpp_quant_blockwise(const void* x, zpp_dtype x_dt, int64_t n, int32_t block,
                               int32_t bits, void* codes, float* scales, cudaStream_t stream) {
  if (!valid_bits(bits) || !valid_block(block) || n < 0 || n > ZPP_MAX_ELEMS)
    return ZPP_ERR_INVALID_ARG;
  if (x_dt != ZPP_F16 && x_dt != ZPP_BF16 && x_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (n == 0) return ZPP_OK;
  if (!x || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (x_dt == ZPP_F32) return ZPP_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_quant(x, x_dt == ZPP_BF16, n, block, bits, codes, scales, stream));
}

zpp_status zpp_dequant_blockwise(const void* codes, const float* scales, int64_t n, int32_t block,
                                 int32_t bits, void* y, zpp_dtype y_dt, cudaStream_t stream) {
  if (!valid_bits(bits) || !valid_block(block) || n < 0 || n > ZPP_MAX_ELEMS)
    return ZPP_ERR_INVALID_ARG;
  if (y_dt != ZPP_F16 && y_dt != ZPP_BF16 && y_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (n == 0) return ZPP_OK;
  if (!codes || !scales || !y) return ZPP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(y, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_dequant(codes, scales, n, block, bits, y, static_cast<int>(y_dt), stream));
}

zpp_status zpp_qgz_reorder_quant_range(const void* grads, zpp_dtype g_dt, int64_t elems_per_rank,
                                       int32_t block, int32_t bits, zpp_topology topo,
                                       zpp_local_range range, void* codes, float* scales,
                                       cudaStream_t stream) {
  int64_t W = 0;
  zpp_status st = check_topology(elems_per_rank, block, bits, topo, &W);
  if (st != ZPP_OK) return st;
  if (g_dt != ZPP_F16 && g_dt != ZPP_BF16 && g_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (!valid_range(range, topo)) return ZPP_ERR_INVALID_ARG;
  if (elems_per_rank == 0 || range.begin == range.end) return ZPP_OK;
  if (!grads || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (g_dt == ZPP_F32) return ZPP_ERR_UNSUPPORTED;
  if (!aligned(grads, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_reorder_quant(grads, g_dt == ZPP_BF16, elems_per_rank, block, bits,
                                             topo.num_nodes, topo.gpus_per_node, range.begin,
                                             range.end, static_cast<int>(W), codes, scales,
                                             stream));
}

zpp_status zpp_qgz_reorder_quant(const void* grads, zpp_dtype g_dt, int64_t elems_per_rank,
                                 int32_t block, int32_t bits, zpp_topology topo, void* codes,
                                 float* scales, cudaStream_t stream) {
  return zpp_qgz_reorder_quant_range(grads, g_dt, elems_per_rank, block, bits, topo,
                                     full_range(topo), codes, scales, stream);
}

zpp_status zpp_qgz_reorder_quant_tensors(const void* const* tensors, const int64_t* sizes,
                                         int32_t num_tensors, zpp_dtype g_dt, int32_t block,
                                         int32_t bits, zpp_topology topo, void* codes,
                                         float* scales, cudaStream_t stream) {
  static_assert(zpp::kMaxTensors == ZPP_MAX_TENSORS, "tensor table size");
  if (!tensors || !sizes || num_tensors < 1 || num_tensors > ZPP_MAX_TENSORS)
    return ZPP_ERR_INVALID_ARG;
  int64_t E = 0;
  for (int32_t t = 0; t < num_tensors; ++t) {
    if (sizes[t] < 0 || sizes[t] >= (int64_t{1} << 31)) return ZPP_ERR_INVALID_ARG;
    E += sizes[t];
    if (E >= (int64_t{1} << 31)) return ZPP_ERR_INVALID_ARG;
  }
  int64_t W = 0;
  zpp_status st = check_topology(E, block, bits, topo, &W);
  if (st != ZPP_OK) return st;
  if (g_dt != ZPP_F16 && g_dt != ZPP_BF16 && g_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (E == 0) return ZPP_OK;
  if (!codes || !scales) return ZPP_ERR_INVALID_ARG;
  for (int32_t t = 0; t < num_tensors; ++t)
    if (sizes[t] > 0 && !tensors[t]) return ZPP_ERR_INVALID_ARG;
  if (g_dt == ZPP_F32) return ZPP_ERR_UNSUPPORTED;
  for (int32_t t = 0; t < num_tensors; ++t)
    if (sizes[t] % 16 != 0 || (sizes[t] > 0 && !aligned(tensors[t], 16))) return ZPP_ERR_MISALIGNED;
  if (!aligned(codes, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  zpp::TensorTable tab;
  tab.count = num_tensors;
  tab.offs[0] = 0;
  for (int32_t t = 0; t < num_tensors; ++t) {
    tab.ptr[t] = static_cast<const uint16_t*>(tensors[t]);
    tab.offs[t + 1] = tab.offs[t] + sizes[t];
  }
  return from_cuda(zpp::launch_reorder_quant_tensors(tab, g_dt == ZPP_BF16, E, block, bits,
                                                     topo.num_nodes, topo.gpus_per_node, codes,
                                                     scales, stream));
}

zpp_status zpp_dequant_reduce_requant_range(const void* codes, const float* scales,
                                            int64_t elems_per_rank, int32_t block, int32_t bits,
                                            zpp_topology topo, zpp_local_range range,
                                            void* out_codes, float* out_scales,
                                            cudaStream_t stream) {
  int64_t W = 0;
  zpp_status st = check_topology(elems_per_rank, block, bits, topo, &W);
  if (st != ZPP_OK) return st;
  if (!valid_range(range, topo)) return ZPP_ERR_INVALID_ARG;
  if (elems_per_rank == 0 || range.begin == range.end) return ZPP_OK;
  if (!codes || !scales || !out_codes || !out_scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out_codes, 16) || !aligned(scales, 4) ||
      !aligned(out_scales, 4))
    return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_dequant_reduce_requant(
      codes, scales, elems_per_rank, elems_per_rank / topo.gpus_per_node, block, bits,
      topo.num_nodes, topo.gpus_per_node, range.begin, range.end, out_codes, out_scales, stream));
}

zpp_status zpp_dequant_reduce_requant(const void* codes, const float* scales,
                                      int64_t elems_per_rank, int32_t block, int32_t bits,
                                      zpp_topology topo, void* out_codes, float* out_scales,
                                      cudaStream_t stream) {
  return zpp_dequant_reduce_requant_range(codes, scales, elems_per_rank, block, bits, topo,
                                          full_range(topo), out_codes, out_scales, stream);
}

zpp_status zpp_dequant_reduce_scaled_range(const void* codes, const float* scales,
                                           int64_t elems_per_rank, int32_t block, int32_t bits,
                                           zpp_topology topo, zpp_local_range range,
                                           float post_scale, void* out, zpp_dtype out_dt,
                                           cudaStream_t stream) {
  int64_t W = 0;
  zpp_status st = check_topology(elems_per_rank, block, bits, topo, &W);
  if (st != ZPP_OK) return st;
  if (out_dt != ZPP_F16 && out_dt != ZPP_BF16 && out_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (!(post_scale == post_scale) || post_scale - post_scale != 0.0f) return ZPP_ERR_INVALID_ARG;
  if (!valid_range(range, topo)) return ZPP_ERR_INVALID_ARG;
  if (elems_per_rank == 0 || range.begin == range.end) return ZPP_OK;
  if (!codes || !scales || !out) return ZPP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_dequant_reduce(
      codes, scales, elems_per_rank / W, elems_per_rank / topo.gpus_per_node, block, bits,
      topo.num_nodes, topo.gpus_per_node, range.begin, range.end, topo.num_nodes, post_scale, out,
      static_cast<int>(out_dt), stream));
}

zpp_status zpp_dequant_reduce_scaled(const void* codes, const float* scales,
                                     int64_t elems_per_rank, int32_t block, int32_t bits,
                                     zpp_topology topo, float post_scale, void* out,
                                     zpp_dtype out_dt, cudaStream_t stream) {
  return zpp_dequant_reduce_scaled_range(codes, scales, elems_per_rank, block, bits, topo,
                                         full_range(topo), post_scale, out, out_dt, stream);
}

zpp_status zpp_dequant_reduce(const void* codes, const float* scales, int64_t elems_per_rank,
                              int32_t block, int32_t bits, zpp_topology topo, float* out,
                              cudaStream_t stream) {
  return zpp_dequant_reduce_scaled_range(codes, scales, elems_per_rank, block, bits, topo,
                                         full_range(topo), 1.0f, out, ZPP_F32, stream);
}

zpp_status zpp_qgz_reorder_quant_local(const void* grads, zpp_dtype g_dt, int64_t elems_per_rank,
                                       int32_t block, int32_t bits, zpp_topology topo,
                                       zpp_local_range range, void* codes, float* scales,
                                       cudaStream_t stream) {
  int64_t W = 0;
  zpp_status st = check_topology(elems_per_rank, block, bits, topo, &W);
  if (st != ZPP_OK) return st;
  if (g_dt != ZPP_F16 && g_dt != ZPP_BF16 && g_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (!valid_range(range, topo)) return ZPP_ERR_INVALID_ARG;
  if (elems_per_rank == 0 || range.begin == range.end) return ZPP_OK;
  if (!grads || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (g_dt == ZPP_F32) return ZPP_ERR_UNSUPPORTED;
  if (!aligned(grads, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_reorder_quant(grads, g_dt == ZPP_BF16, elems_per_rank, block, bits,
                                             topo.num_nodes, topo.gpus_per_node, range.begin,
                                             range.end, 1, codes, scales, stream));
}

namespace {
// Checks shared by the two calls on received chunks: `len` elements per source, a
// multiple of the block, `sources` of them.
zpp_status check_received(int64_t len, int32_t block, int32_t bits, int32_t sources) {
  if (!valid_bits(bits) || !valid_block(block)) return ZPP_ERR_INVALID_ARG;
  if (sources < 1 || sources > 65535) return ZPP_ERR_INVALID_ARG;
  if (len < 0 || len >= (int64_t{1} << 31) || len % block != 0) return ZPP_ERR_INVALID_ARG;
  if (len * sources > ZPP_MAX_ELEMS) return ZPP_ERR_INVALID_ARG;
  return ZPP_OK;
}
}  // namespace

zpp_status zpp_dequant_reduce_requant_local(const void* codes, const float* scales, int64_t chunk,
                                            int32_t block, int32_t bits, int32_t sources,
                                            void* out_codes, float* out_scales,
                                            cudaStream_t stream) {
  const zpp_status st = check_received(chunk, block, bits, sources);
  if (st != ZPP_OK) return st;
  if (chunk == 0) return ZPP_OK;
  if (!codes || !scales || !out_codes || !out_scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out_codes, 16) || !aligned(scales, 4) ||
      !aligned(out_scales, 4))
    return ZPP_ERR_MISALIGNED;
  // one receiver (N = 1, l = 0) whose sources are the received chunks, `chunk` apart
  return from_cuda(zpp::launch_dequant_reduce_requant(codes, scales, chunk, chunk, block, bits, 1,
                                                      sources, 0, 1, out_codes, out_scales,
                                                      stream));
}

zpp_status zpp_dequant_reduce_local(const void* codes, const float* scales, int64_t slice,
                                    int32_t block, int32_t bits, int32_t sources,
                                    float post_scale, void* out, zpp_dtype out_dt,
                                    cudaStream_t stream) {
  const zpp_status st = check_received(slice, block, bits, sources);
  if (st != ZPP_OK) return st;
  if (out_dt != ZPP_F16 && out_dt != ZPP_BF16 && out_dt != ZPP_F32) return ZPP_ERR_INVALID_ARG;
  if (!(post_scale == post_scale) || post_scale - post_scale != 0.0f) return ZPP_ERR_INVALID_ARG;
  if (slice == 0) return ZPP_OK;
  if (!codes || !scales || !out) return ZPP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out, 16) || !aligned(scales, 4)) return ZPP_ERR_MISALIGNED;
  // one receiver (n = 0, l = 0) whose N sources are the received slices, `slice` apart
  return from_cuda(zpp::launch_dequant_reduce(codes, scales, slice, slice, block, bits, sources, 1,
                                              0, 1, 1, post_scale, out, static_cast<int>(out_dt),
                                              stream));
}

zpp_status zpp_device_fault(uint32_t* flags, int32_t clear) {
  if (!flags) return ZPP_ERR_INVALID_ARG;
  unsigned v = 0;
  const zpp_status st = from_cuda(zpp::read_device_fault(&v, clear != 0));
  *flags = st == ZPP_OK ? v : 0u;
  return st;
}

zpp_status zpp_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return ZPP_ERR_INVALID_ARG;
  return from_cuda(zpp::launch_wait_selftest(limit_ns, stream));
}

zpp_status zpp_device_copy(const void* src, void* dst, int64_t bytes, cudaStream_t stream) {
  if (bytes < 0 || bytes % 32 != 0) return ZPP_ERR_INVALID_ARG;
  if (bytes == 0) return ZPP_OK;
  if (!src || !dst) return ZPP_ERR_INVALID_ARG;
  if (!aligned(src, 32) || !aligned(dst, 32)) return ZPP_ERR_MISALIGNED;
  return from_cuda(zpp::launch_copy(src, dst, bytes, stream));
}

}  // extern "C"
