"""ctypes binding of ``libzpp.so`` (argument marshalling only).

The raw functions carry the C names and take device addresses as integers; the tensor
helpers below allocate outputs with torch on the input's device, pass pointers and the
current CUDA stream, and raise on a non-OK status. Every step of the computation runs
in the library's kernels: there is no CPU path, and a missing library or a CPU tensor
is an error.
"""
import ctypes
import os
import re

from . import build as _build

ZPP_OK, ZPP_ERR_INVALID_ARG, ZPP_ERR_MISALIGNED, ZPP_ERR_UNSUPPORTED, ZPP_ERR_CUDA = range(5)
ZPP_F16, ZPP_BF16, ZPP_F32 = 0, 1, 2

HEADER = os.path.join(_build.ROOT, "include", "zpp.h")


class Topology(ctypes.Structure):
    _fields_ = [("num_nodes", ctypes.c_int32), ("gpus_per_node", ctypes.c_int32)]


class LocalRange(ctypes.Structure):
    _fields_ = [("begin", ctypes.c_int32), ("end", ctypes.c_int32)]


class ZppError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {zpp_status_string(status)}")


_lib = None


def lib_path():
    return _build.LIB


def lib():
    """Load libzpp.so (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: build it with __graft_entry__.build() "
                           "(there is no fallback path)")
    L = ctypes.CDLL(_build.LIB)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    sig = {
        "zpp_quant_blockwise": [vp, i32, i64, i32, i32, vp, vp, vp],
        "zpp_dequant_blockwise": [vp, vp, i64, i32, i32, vp, i32, vp],
        "zpp_qgz_reorder_quant": [vp, i32, i64, i32, i32, Topology, vp, vp, vp],
        "zpp_dequant_reduce_requant": [vp, vp, i64, i32, i32, Topology, vp, vp, vp],
        "zpp_dequant_reduce": [vp, vp, i64, i32, i32, Topology, vp, vp],
        "zpp_dequant_reduce_scaled": [vp, vp, i64, i32, i32, Topology, ctypes.c_float, vp, i32,
                                      vp],
        "zpp_qgz_reorder_quant_range": [vp, i32, i64, i32, i32, Topology, LocalRange, vp, vp, vp],
        "zpp_qgz_reorder_quant_tensors": [vp, vp, i32, i32, i32, i32, Topology, vp, vp, vp],
        "zpp_dequant_reduce_requant_range": [vp, vp, i64, i32, i32, Topology, LocalRange, vp, vp,
                                             vp],
        "zpp_dequant_reduce_scaled_range": [vp, vp, i64, i32, i32, Topology, LocalRange,
                                            ctypes.c_float, vp, i32, vp],
        "zpp_device_copy": [vp, vp, i64, vp],
        "zpp_qgz_reorder_quant_local": [vp, i32, i64, i32, i32, Topology, LocalRange, vp, vp,
                                        vp],
        "zpp_dequant_reduce_requant_local": [vp, vp, i64, i32, i32, i32, vp, vp, vp],
        "zpp_dequant_reduce_local": [vp, vp, i64, i32, i32, i32, ctypes.c_float, vp, i32, vp],
        "zpp_device_fault": [ctypes.POINTER(ctypes.c_uint32), i32],
        "zpp_wait_selftest": [ctypes.c_uint64, vp],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.zpp_code_bytes.argtypes = [i64, i32]
    L.zpp_code_bytes.restype = i64
    L.zpp_num_scales.argtypes = [i64, i32]
    L.zpp_num_scales.restype = i64
    L.zpp_status_string.argtypes = [ctypes.c_int]
    L.zpp_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def declared_symbols(header=HEADER):
    """Names of the functions the public header declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"ZPP_API\s+[\w\s\*]*?\b(zpp_\w+)\s*\(", text)))


# ----------------------------------------------------------------------------- raw ABI
def zpp_quant_blockwise(x, x_dt, n, block, bits, codes, scales, stream=0):
    return lib().zpp_quant_blockwise(x, x_dt, n, block, bits, codes, scales, stream)


def zpp_dequant_blockwise(codes, scales, n, block, bits, y, y_dt, stream=0):
    return lib().zpp_dequant_blockwise(codes, scales, n, block, bits, y, y_dt, stream)


def zpp_qgz_reorder_quant(grads, g_dt, elems_per_rank, block, bits, topo, codes, scales, stream=0):
    return lib().zpp_qgz_reorder_quant(grads, g_dt, elems_per_rank, block, bits, topo, codes,
                                       scales, stream)


def zpp_qgz_reorder_quant_tensors(tensor_ptrs, sizes, g_dt, block, bits, topo, codes, scales,
                                  stream=0):
    """tensor_ptrs, sizes: Python sequences (marshalled into host arrays for the call)."""
    T = len(tensor_ptrs)
    ptrs = (ctypes.c_void_p * max(T, 1))(*tensor_ptrs)
    lens = (ctypes.c_int64 * max(T, 1))(*sizes)
    return lib().zpp_qgz_reorder_quant_tensors(ptrs, lens, T, g_dt, block, bits, topo, codes,
                                               scales, stream)


def zpp_dequant_reduce_requant(codes, scales, elems_per_rank, block, bits, topo, out_codes,
                               out_scales, stream=0):
    return lib().zpp_dequant_reduce_requant(codes, scales, elems_per_rank, block, bits, topo,
                                            out_codes, out_scales, stream)


def zpp_dequant_reduce(codes, scales, elems_per_rank, block, bits, topo, out, stream=0):
    return lib().zpp_dequant_reduce(codes, scales, elems_per_rank, block, bits, topo, out, stream)


def zpp_dequant_reduce_scaled(codes, scales, elems_per_rank, block, bits, topo, post_scale, out,
                              out_dt, stream=0):
    return lib().zpp_dequant_reduce_scaled(codes, scales, elems_per_rank, block, bits, topo,
                                           post_scale, out, out_dt, stream)


def zpp_qgz_reorder_quant_range(grads, g_dt, elems_per_rank, block, bits, topo, rng, codes,
                                scales, stream=0):
    return lib().zpp_qgz_reorder_quant_range(grads, g_dt, elems_per_rank, block, bits, topo, rng,
                                             codes, scales, stream)


def zpp_dequant_reduce_requant_range(codes, scales, elems_per_rank, block, bits, topo, rng,
                                     out_codes, out_scales, stream=0):
    return lib().zpp_dequant_reduce_requant_range(codes, scales, elems_per_rank, block, bits,
                                                  topo, rng, out_codes, out_scales, stream)


def zpp_dequant_reduce_scaled_range(codes, scales, elems_per_rank, block, bits, topo, rng,
                                    post_scale, out, out_dt, stream=0):
    return lib().zpp_dequant_reduce_scaled_range(codes, scales, elems_per_rank, block, bits,
                                                 topo, rng, post_scale, out, out_dt, stream)


def zpp_qgz_reorder_quant_local(grads, g_dt, elems_per_rank, block, bits, topo, rng, codes,
                                scales, stream=0):
    return lib().zpp_qgz_reorder_quant_local(grads, g_dt, elems_per_rank, block, bits, topo, rng,
                                             codes, scales, stream)


def zpp_dequant_reduce_requant_local(codes, scales, chunk, block, bits, sources, out_codes,
                                     out_scales, stream=0):
    return lib().zpp_dequant_reduce_requant_local(codes, scales, chunk, block, bits, sources,
                                                  out_codes, out_scales, stream)


def zpp_dequant_reduce_local(codes, scales, slice_len, block, bits, sources, post_scale, out,
                             out_dt, stream=0):
    return lib().zpp_dequant_reduce_local(codes, scales, slice_len, block, bits, sources,
                                          post_scale, out, out_dt, stream)


def zpp_device_copy(src, dst, nbytes, stream=0):
    return lib().zpp_device_copy(src, dst, nbytes, stream)


def zpp_device_fault(clear=False):
    """The device fault word (see include/zpp.h); synchronises with the device."""
    v = ctypes.c_uint32(0)
    _check(lib().zpp_device_fault(ctypes.byref(v), 1 if clear else 0), "zpp_device_fault")
    return int(v.value)


def zpp_wait_selftest(limit_ns, stream=0):
    return lib().zpp_wait_selftest(limit_ns, stream)


def zpp_code_bytes(n, bits):
    return int(lib().zpp_code_bytes(n, bits))


def zpp_num_scales(n, block):
    return int(lib().zpp_num_scales(n, block))


def zpp_status_string(status):
    return lib().zpp_status_string(int(status)).decode()


# ----------------------------------------------------------------------------- tensors
# The wrappers below check every tensor's element count and dtype against what the call
# reads or writes, then that all tensors are contiguous CUDA tensors on one device, and
# raise ValueError before calling into libzpp. Sizes that the C ABI itself rejects (bad
# bits, block or topology) are left to it and raise ZppError with its status.
def _torch():
    import torch
    return torch


def _dt(t):
    torch = _torch()
    return {torch.float16: ZPP_F16, torch.bfloat16: ZPP_BF16, torch.float32: ZPP_F32}[t]


def _bytes_dtypes():
    torch = _torch()
    return (torch.uint8, torch.int8)


def _need(t, name, numel=None, dtypes=None):
    """t must hold exactly `numel` elements of one of `dtypes` (None: not checked)."""
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected one of {tuple(dtypes)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")


def _cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("zpp operates on CUDA tensors only (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("zpp needs contiguous tensors")
    if any(t.device != ts[0].device for t in ts):
        raise ValueError("all tensors of a call must be on one device")


def _stream(t):
    return _torch().cuda.current_stream(t.device).cuda_stream


def _check(status, where):
    if status != ZPP_OK:
        raise ZppError(status, where)


def _sizes_ok(n, block, bits):
    return n >= 0 and bits in (4, 8) and block in (64, 128, 256, 512, 1024, 2048, 4096)


def _qgz_sizes(E, block, bits, N, M):
    """(W, C, S) when E fits the topology (else None: the C ABI reports it)."""
    W = N * M
    if N < 1 or M < 1 or not _sizes_ok(E, block, bits) or E % (W * block):
        return None
    return W, E // M, E // W


def quant_blockwise(x, block, bits, codes=None, scales=None):
    """x (fp16/bf16, any shape) -> (codes uint8[code_bytes], scales fp32[num_scales])."""
    torch = _torch()
    n = x.numel()
    _need(x, "x", dtypes=(torch.float16, torch.bfloat16))
    ok = _sizes_ok(n, block, bits)
    if codes is not None:
        _need(codes, "codes", zpp_code_bytes(n, bits) if ok else None, _bytes_dtypes())
    if scales is not None:
        _need(scales, "scales", zpp_num_scales(n, block) if ok else None, (torch.float32,))
    _cuda(x, *(t for t in (codes, scales) if t is not None))
    if codes is None:
        codes = torch.empty(max(zpp_code_bytes(n, bits), 0), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(max(zpp_num_scales(n, block), 0), dtype=torch.float32,
                             device=x.device)
    _check(zpp_quant_blockwise(x.data_ptr(), _dt(x.dtype), n, block, bits, codes.data_ptr(),
                               scales.data_ptr(), _stream(x)), "zpp_quant_blockwise")
    return codes, scales


def dequant_blockwise(codes, scales, n, block, bits, dtype=None, y=None):
    """codes, scales -> y[n] of `dtype` (default fp16)."""
    torch = _torch()
    ok = _sizes_ok(n, block, bits)
    _need(codes, "codes", zpp_code_bytes(n, bits) if ok else None, _bytes_dtypes())
    _need(scales, "scales", zpp_num_scales(n, block) if ok else None, (torch.float32,))
    if y is not None:
        _need(y, "y", n, (torch.float16, torch.bfloat16, torch.float32))
    _cuda(codes, scales, *(t for t in (y,) if t is not None))
    if y is None:
        y = torch.empty(max(n, 0), dtype=dtype or torch.float16, device=codes.device)
    _check(zpp_dequant_blockwise(codes.data_ptr(), scales.data_ptr(), n, block, bits,
                                 y.data_ptr(), _dt(y.dtype), _stream(codes)),
           "zpp_dequant_blockwise")
    return y


def qgz_reorder_quant(grads, block, bits, N, M, codes=None, scales=None):
    """grads [W][E] (fp16/bf16) -> (codes uint8 [W][code_bytes(E)], scales fp32 [W][E/block])."""
    torch = _torch()
    W = N * M
    _need(grads, "grads", dtypes=(torch.float16, torch.bfloat16))
    if W < 1 or grads.numel() % W:
        raise ValueError(f"grads: {grads.numel()} elements do not split into {W} ranks")
    E = grads.numel() // W
    sz = _qgz_sizes(E, block, bits, N, M)
    if codes is not None:
        _need(codes, "codes", W * zpp_code_bytes(E, bits) if sz else None, _bytes_dtypes())
    if scales is not None:
        _need(scales, "scales", W * (E // block) if sz else None, (torch.float32,))
    _cuda(grads, *(t for t in (codes, scales) if t is not None))
    if codes is None:
        codes = torch.empty((W, max(zpp_code_bytes(E, bits), 0)), dtype=torch.uint8,
                            device=grads.device)
    if scales is None:
        scales = torch.empty((W, E // block if block > 0 else 0), dtype=torch.float32,
                             device=grads.device)
    _check(zpp_qgz_reorder_quant(grads.data_ptr(), _dt(grads.dtype), E, block, bits,
                                 Topology(N, M), codes.data_ptr(), scales.data_ptr(),
                                 _stream(grads)), "zpp_qgz_reorder_quant")
    return codes, scales


def qgz_reorder_quant_tensors(tensors, block, bits, N, M, codes=None, scales=None):
    """The bucket given as a list of gradient tensors, tensor t of shape [W][n_t] (the W
    ranks' copies; any shape with W * n_t elements, contiguous) -> the codes and scales
    qgz_reorder_quant gives for the bucket whose rank r concatenates row r of every tensor."""
    torch = _torch()
    if not tensors:
        raise ValueError("qgz_reorder_quant_tensors needs at least one tensor")
    W = N * M
    dt = tensors[0].dtype
    for i, t in enumerate(tensors):
        _need(t, f"tensors[{i}]", dtypes=(dt,))
    _need(tensors[0], "tensors[0]", dtypes=(torch.float16, torch.bfloat16))
    if W < 1 or any(t.numel() % W for t in tensors):
        raise ValueError("every tensor holds W equal per-rank copies")
    sizes = [t.numel() // W for t in tensors]
    E = sum(sizes)
    sz = _qgz_sizes(E, block, bits, N, M)
    if codes is not None:
        _need(codes, "codes", W * zpp_code_bytes(E, bits) if sz else None, _bytes_dtypes())
    if scales is not None:
        _need(scales, "scales", W * (E // block) if sz else None, (torch.float32,))
    _cuda(*tensors, *(t for t in (codes, scales) if t is not None))
    dev = tensors[0].device
    if codes is None:
        codes = torch.empty((W, max(zpp_code_bytes(E, bits), 0)), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((W, E // block if block > 0 else 0), dtype=torch.float32, device=dev)
    _check(zpp_qgz_reorder_quant_tensors([t.data_ptr() for t in tensors], sizes, _dt(dt), block,
                                         bits, Topology(N, M), codes.data_ptr(), scales.data_ptr(),
                                         _stream(tensors[0])), "zpp_qgz_reorder_quant_tensors")
    return codes, scales


def _hop_inputs(codes, scales, E, block, bits, N, M, hop):
    """Checks the codes / scales a hop reads: hop 1 reads the step-1 buffers ([W][E]
    elements per rank), hop 2 the hop-1 buffers ([W][C], C = E / M)."""
    torch = _torch()
    sz = _qgz_sizes(E, block, bits, N, M)
    n = None if sz is None else (E if hop == 1 else sz[1])
    W = N * M
    _need(codes, "codes", W * zpp_code_bytes(n, bits) if sz else None, _bytes_dtypes())
    _need(scales, "scales", W * (n // block) if sz else None, (torch.float32,))
    return sz


def dequant_reduce_requant(codes, scales, E, block, bits, N, M, out_codes=None, out_scales=None):
    """Intra-node hop -> (codes uint8 [W][code_bytes(E/M)], scales fp32 [W][E/M/block])."""
    torch = _torch()
    sz = _hop_inputs(codes, scales, E, block, bits, N, M, hop=1)
    W, C = N * M, E // M if M > 0 else 0
    if out_codes is not None:
        _need(out_codes, "out_codes", W * zpp_code_bytes(C, bits) if sz else None,
              _bytes_dtypes())
    if out_scales is not None:
        _need(out_scales, "out_scales", W * (C // block) if sz else None, (torch.float32,))
    _cuda(codes, scales, *(t for t in (out_codes, out_scales) if t is not None))
    if out_codes is None:
        out_codes = torch.empty((W, max(zpp_code_bytes(C, bits), 0)), dtype=torch.uint8,
                                device=codes.device)
    if out_scales is None:
        out_scales = torch.empty((W, C // block if block > 0 else 0), dtype=torch.float32,
                                 device=codes.device)
    _check(zpp_dequant_reduce_requant(codes.data_ptr(), scales.data_ptr(), E, block, bits,
                                      Topology(N, M), out_codes.data_ptr(), out_scales.data_ptr(),
                                      _stream(codes)), "zpp_dequant_reduce_requant")
    return out_codes, out_scales


def dequant_reduce(codes, scales, E, block, bits, N, M, out=None):
    """Inter-node hop -> fp32 [W][E/W], each rank's summed owner slice."""
    torch = _torch()
    sz = _hop_inputs(codes, scales, E, block, bits, N, M, hop=2)
    W = N * M
    if out is not None:
        _need(out, "out", W * (E // W) if sz else None, (torch.float32,))
    _cuda(codes, scales, *(t for t in (out,) if t is not None))
    if out is None:
        out = torch.empty((W, E // W if W > 0 else 0), dtype=torch.float32, device=codes.device)
    _check(zpp_dequant_reduce(codes.data_ptr(), scales.data_ptr(), E, block, bits, Topology(N, M),
                              out.data_ptr(), _stream(codes)), "zpp_dequant_reduce")
    return out


def dequant_reduce_scaled(codes, scales, E, block, bits, N, M, post_scale=None, dtype=None,
                          out=None):
    """Inter-node hop with the average folded in: [W][E/W] of `dtype` (default fp32) holding
    fp32(sum * post_scale); post_scale defaults to 1/W (the average over ranks)."""
    torch = _torch()
    sz = _hop_inputs(codes, scales, E, block, bits, N, M, hop=2)
    W = N * M
    if out is not None:
        _need(out, "out", W * (E // W) if sz else None,
              (torch.float16, torch.bfloat16, torch.float32))
    _cuda(codes, scales, *(t for t in (out,) if t is not None))
    if post_scale is None:
        post_scale = 1.0 / W
    if out is None:
        out = torch.empty((W, E // W if W > 0 else 0), dtype=dtype or torch.float32,
                          device=codes.device)
    _check(zpp_dequant_reduce_scaled(codes.data_ptr(), scales.data_ptr(), E, block, bits,
                                     Topology(N, M), float(post_scale), out.data_ptr(),
                                     _dt(out.dtype), _stream(codes)), "zpp_dequant_reduce_scaled")
    return out


# ------------------------------------------------------------------ one real rank's steps
def qgz_reorder_quant_local(grads, block, bits, N, M, codes=None, scales=None, chunks=None):
    """This rank's gradient bucket [E] (fp16/bf16) -> its reordered codes [code_bytes(E)]
    and scales [E/block]: chunk l' (N*S elements) goes to local peer l' in hop 1. With
    `chunks` = (begin, end) only those chunks are written (into the given buffers)."""
    torch = _torch()
    _need(grads, "grads", dtypes=(torch.float16, torch.bfloat16))
    E = grads.numel()
    sz = _qgz_sizes(E, block, bits, N, M)
    if codes is not None:
        _need(codes, "codes", zpp_code_bytes(E, bits) if sz else None, _bytes_dtypes())
    if scales is not None:
        _need(scales, "scales", E // block if sz else None, (torch.float32,))
    _cuda(grads, *(t for t in (codes, scales) if t is not None))
    if codes is None:
        codes = torch.empty(max(zpp_code_bytes(E, bits), 0), dtype=torch.uint8, device=grads.device)
    if scales is None:
        scales = torch.empty(E // block if block > 0 else 0, dtype=torch.float32,
                             device=grads.device)
    rng = LocalRange(*(chunks if chunks is not None else (0, M)))
    _check(zpp_qgz_reorder_quant_local(grads.data_ptr(), _dt(grads.dtype), E, block, bits,
                                       Topology(N, M), rng, codes.data_ptr(), scales.data_ptr(),
                                       _stream(grads)), "zpp_qgz_reorder_quant_local")
    return codes, scales


def _received(codes, scales, sources, length, block, bits):
    torch = _torch()
    ok = sources >= 1 and _sizes_ok(length, block, bits) and length % block == 0
    _need(codes, "codes", sources * zpp_code_bytes(length, bits) if ok else None, _bytes_dtypes())
    _need(scales, "scales", sources * (length // block) if ok else None, (torch.float32,))
    return ok


def dequant_reduce_requant_local(codes, scales, chunk, block, bits, sources, out_codes=None,
                                 out_scales=None):
    """The fused intra-node hop on the chunks this rank received ([sources][chunk] codes and
    scales, sources in local-index order) -> its hop-1 codes [code_bytes(chunk)] and scales."""
    torch = _torch()
    ok = _received(codes, scales, sources, chunk, block, bits)
    if out_codes is not None:
        _need(out_codes, "out_codes", zpp_code_bytes(chunk, bits) if ok else None, _bytes_dtypes())
    if out_scales is not None:
        _need(out_scales, "out_scales", chunk // block if ok else None, (torch.float32,))
    _cuda(codes, scales, *(t for t in (out_codes, out_scales) if t is not None))
    if out_codes is None:
        out_codes = torch.empty(max(zpp_code_bytes(chunk, bits), 0), dtype=torch.uint8,
                                device=codes.device)
    if out_scales is None:
        out_scales = torch.empty(chunk // block if block > 0 else 0, dtype=torch.float32,
                                 device=codes.device)
    _check(zpp_dequant_reduce_requant_local(codes.data_ptr(), scales.data_ptr(), chunk, block,
                                            bits, sources, out_codes.data_ptr(),
                                            out_scales.data_ptr(), _stream(codes)),
           "zpp_dequant_reduce_requant_local")
    return out_codes, out_scales


def dequant_reduce_local(codes, scales, slice_len, block, bits, sources, post_scale=1.0,
                         dtype=None, out=None):
    """The final inter-node hop on the slices this rank received ([sources][slice_len],
    nodes in ascending order) -> its owner slice [slice_len] of `dtype` (default fp32),
    fp32(sum * post_scale)."""
    torch = _torch()
    ok = _received(codes, scales, sources, slice_len, block, bits)
    if out is not None:
        _need(out, "out", slice_len if ok else None, (torch.float16, torch.bfloat16, torch.float32))
    _cuda(codes, scales, *(t for t in (out,) if t is not None))
    if out is None:
        out = torch.empty(max(slice_len, 0), dtype=dtype or torch.float32, device=codes.device)
    _check(zpp_dequant_reduce_local(codes.data_ptr(), scales.data_ptr(), slice_len, block, bits,
                                    sources, float(post_scale), out.data_ptr(), _dt(out.dtype),
                                    _stream(codes)), "zpp_dequant_reduce_local")
    return out


class QgzBuffers:
    """Device buffers of one qgZ exchange: reordered codes/scales (c0, s0), hop-1
    codes/scales (c1, s1) and the owner slices (out)."""

    def __init__(self, c0, s0, c1, s1, out):
        self.c0, self.s0, self.c1, self.s1, self.out = c0, s0, c1, s1, out

    @classmethod
    def allocate(cls, W, E, block, bits, M, device, out_dtype=None):
        torch = _torch()
        C = E // M
        return cls(torch.empty((W, zpp_code_bytes(E, bits)), dtype=torch.uint8, device=device),
                   torch.empty((W, E // block), dtype=torch.float32, device=device),
                   torch.empty((W, zpp_code_bytes(C, bits)), dtype=torch.uint8, device=device),
                   torch.empty((W, C // block), dtype=torch.float32, device=device),
                   torch.empty((W, E // W), dtype=out_dtype or torch.float32, device=device))

    def check(self, W, E, block, bits, M):
        """Raise ValueError unless every buffer has the size and dtype of an exchange of W
        ranks of E elements (the layouts of allocate())."""
        torch = _torch()
        C = E // M
        _need(self.c0, "bufs.c0", W * zpp_code_bytes(E, bits), _bytes_dtypes())
        _need(self.s0, "bufs.s0", W * (E // block), (torch.float32,))
        _need(self.c1, "bufs.c1", W * zpp_code_bytes(C, bits), _bytes_dtypes())
        _need(self.s1, "bufs.s1", W * (C // block), (torch.float32,))
        _need(self.out, "bufs.out", W * (E // W), (torch.float16, torch.bfloat16, torch.float32))


def qgz_pipelined(grads, block, bits, N, M, post_scale=1.0, bufs=None, streams=None,
                  n_streams=2, chunks=None):
    """The whole qgZ exchange as independent local-index sub-pipelines (reorder + quantise
    of chunks l, hop 1 for receivers (n, l), hop 2 for ranks (n, l)), joined back into the
    caller's stream. `chunks` local indices form one sub-pipeline (default: one per l).

    Schedules: with a list of `streams`, whole sub-pipelines go round robin over them;
    with ``streams=("split", low, high)`` every reorder + quantise runs on the `low`
    stream and each sub-pipeline's two hops on the `high` stream, gated by an event, so
    hop work fills the SMs that reorder work frees (give `high` the higher priority).
    Returns the buffers (owner slices in ``bufs.out``; fp32 by default)."""
    torch = _torch()
    W = N * M
    _need(grads, "grads", dtypes=(torch.float16, torch.bfloat16))
    if W < 1 or grads.numel() % W:
        raise ValueError(f"grads: {grads.numel()} elements do not split into {W} ranks")
    E = grads.numel() // W
    if _qgz_sizes(E, block, bits, N, M) is None:
        raise ValueError("elements per rank must be a multiple of W * block (bits 4 or 8, "
                         "block a power of two in [64, 4096])")
    if bufs is not None:
        bufs.check(W, E, block, bits, M)
        _cuda(grads, bufs.c0, bufs.s0, bufs.c1, bufs.s1, bufs.out)
    else:
        _cuda(grads)
        bufs = QgzBuffers.allocate(W, E, block, bits, M, grads.device)
    main = torch.cuda.current_stream(grads.device)
    if streams is None:
        streams = [torch.cuda.Stream(grads.device) for _ in range(min(n_streams, M))]
    split = len(streams) == 3 and streams[0] == "split"
    side = list(streams[1:]) if split else list(streams)
    chunks = chunks or 1
    fork = torch.cuda.Event()
    fork.record(main)
    topo = Topology(N, M)
    gdt, odt = _dt(grads.dtype), _dt(bufs.out.dtype)
    for st in side:
        st.wait_event(fork)
    for i, l0 in enumerate(range(0, M, chunks)):
        rng = LocalRange(l0, min(M, l0 + chunks))
        st_q = side[0] if split else side[i % len(side)]
        st_h = side[1] if split else st_q
        _check(zpp_qgz_reorder_quant_range(grads.data_ptr(), gdt, E, block, bits, topo, rng,
                                           bufs.c0.data_ptr(), bufs.s0.data_ptr(),
                                           st_q.cuda_stream), "zpp_qgz_reorder_quant_range")
        if split:
            ready = torch.cuda.Event()
            ready.record(st_q)
            st_h.wait_event(ready)
        _check(zpp_dequant_reduce_requant_range(bufs.c0.data_ptr(), bufs.s0.data_ptr(), E, block,
                                                bits, topo, rng, bufs.c1.data_ptr(),
                                                bufs.s1.data_ptr(), st_h.cuda_stream),
               "zpp_dequant_reduce_requant_range")
        _check(zpp_dequant_reduce_scaled_range(bufs.c1.data_ptr(), bufs.s1.data_ptr(), E, block,
                                               bits, topo, rng, float(post_scale),
                                               bufs.out.data_ptr(), odt, st_h.cuda_stream),
               "zpp_dequant_reduce_scaled_range")
    for st in side:
        join = torch.cuda.Event()
        join.record(st)
        main.wait_event(join)
    return bufs


def device_copy(src, dst):
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() < nbytes:
        raise ValueError(f"dst holds {dst.numel() * dst.element_size()} bytes, src {nbytes}")
    _cuda(src, dst)
    _check(zpp_device_copy(src.data_ptr(), dst.data_ptr(), nbytes, _stream(src)), "zpp_device_copy")
    return dst
