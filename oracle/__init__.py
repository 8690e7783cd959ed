"""Python handle on the CPU oracle (``oracle/zpp_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by
the CPU-baseline / reference legs of ``bench.py``; never by the product package. It
takes and returns numpy arrays. fp16 and bf16 data travel as ``uint16`` bit patterns.

Parity pins: see ``tests/test_oracle_pins.py`` (every function here is pinned there by
closed forms, invariants, brute force or hand-derived fixtures; none is "parity unpinned").
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16, BF16, F32 = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        vp = ctypes.c_void_p
        L.or_set_threads.argtypes = [i32]
        L.or_set_threads.restype = i32
        L.or_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.or_f16_to_f32.restype = ctypes.c_float
        L.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_f32.restype = ctypes.c_float
        L.or_f32_to_f16.argtypes = [ctypes.c_float]
        L.or_f32_to_f16.restype = ctypes.c_uint16
        L.or_f32_to_bf16.argtypes = [ctypes.c_float]
        L.or_f32_to_bf16.restype = ctypes.c_uint16
        L.or_code_bytes.argtypes = [i64, i32]
        L.or_code_bytes.restype = i64
        L.or_quant_blockwise.argtypes = [vp, i32, i64, i64, i32, vp, vp]
        L.or_dequant_blockwise.argtypes = [vp, vp, i64, i64, i32, vp, i32]
        L.or_reorder_position.argtypes = [i64, i32, i32]
        L.or_reorder_position.restype = i64
        L.or_reorder_slices.argtypes = [vp, i64, i32, i32, vp]
        L.or_qgz_reorder_quant.argtypes = [vp, i32, i64, i64, i32, i32, i32, vp, vp]
        L.or_dequant_reduce_requant.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp]
        L.or_dequant_reduce.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp]
        L.or_qgz_passthrough.argtypes = [vp, i64, i32, i32, i32, vp]
        L.or_dequant_reduce_scaled.argtypes = [vp, vp, i64, i64, i32, i32, i32, ctypes.c_float,
                                               vp, i32]
        L.or_dequant_reduce_requant_chunks.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp]
        L.or_dequant_reduce_chunks.argtypes = [vp, vp, i64, i64, i32, i32, ctypes.c_float, vp,
                                               i32]
        for name in ("or_quant_blockwise", "or_dequant_blockwise", "or_qgz_reorder_quant",
                     "or_dequant_reduce_requant", "or_dequant_reduce", "or_qgz_passthrough",
                     "or_dequant_reduce_scaled", "or_dequant_reduce_requant_chunks",
                     "or_dequant_reduce_chunks", "or_rounding_is_nearest"):
            getattr(L, name).restype = i32
        if not L.or_rounding_is_nearest():
            raise RuntimeError("oracle requires round-to-nearest floating-point mode")
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _contig(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _value_dtype(dt):
    return np.float32 if dt == F32 else np.uint16


def set_threads(n: int) -> int:
    """Set the OpenMP thread count (0 keeps it); return the count in use."""
    return int(lib().or_set_threads(int(n)))


def code_bytes(n: int, bits: int) -> int:
    return int(lib().or_code_bytes(int(n), int(bits)))


def num_scales(n: int, block: int) -> int:
    return (int(n) + int(block) - 1) // int(block)


def f16_to_f32(h: int) -> float:
    return lib().or_f16_to_f32(int(h))


def bf16_to_f32(b: int) -> float:
    return lib().or_bf16_to_f32(int(b))


def f32_to_f16(f) -> int:
    return int(lib().or_f32_to_f16(float(np.float32(f))))


def f32_to_bf16(f) -> int:
    return int(lib().or_f32_to_bf16(float(np.float32(f))))


def quant_blockwise(x, dtype: int, block: int, bits: int):
    """Block-wise symmetric quantisation. x: uint16 bits (fp16/bf16) or float32.
    Returns (codes uint8[code_bytes(n)], scales float32[ceil(n/block)])."""
    x = _contig(x, _value_dtype(dtype)).reshape(-1)
    n = x.size
    codes = np.zeros(code_bytes(n, bits), np.uint8)
    scales = np.zeros(num_scales(n, block), np.float32)
    if n and lib().or_quant_blockwise(_p(x), dtype, n, block, bits, _p(codes), _p(scales)):
        raise MemoryError("oracle quant failed")
    return codes, scales


def dequant_blockwise(codes, scales, n: int, block: int, bits: int, y_dtype: int):
    """codes x scale -> y (uint16 bits for fp16/bf16, float32 for fp32)."""
    codes = _contig(codes, np.uint8).reshape(-1)
    scales = _contig(scales, np.float32).reshape(-1)
    assert codes.size >= code_bytes(n, bits) and scales.size >= num_scales(n, block)
    y = np.zeros(n, _value_dtype(y_dtype))
    if n:
        lib().or_dequant_blockwise(_p(codes), _p(scales), n, block, bits, _p(y), y_dtype)
    return y


def reorder_position(j: int, N: int, M: int) -> int:
    return int(lib().or_reorder_position(int(j), int(N), int(M)))


def reorder_slices(src, N: int, M: int):
    src = _contig(src, np.float32).reshape(-1)
    dst = np.empty_like(src)
    lib().or_reorder_slices(_p(src), src.size, N, M, _p(dst))
    return dst


def _check_topo(E, block, N, M):
    W = N * M
    if E % (W * block):
        raise ValueError("elements per rank must be a multiple of W*block")


def qgz_reorder_quant(grads, dtype: int, block: int, bits: int, N: int, M: int):
    """grads [W][E] -> (codes uint8 [W][code_bytes(E)], scales float32 [W][E/block])."""
    W = N * M
    grads = _contig(grads, _value_dtype(dtype)).reshape(W, -1)
    E = grads.shape[1]
    _check_topo(E, block, N, M)
    codes = np.zeros((W, code_bytes(E, bits)), np.uint8)
    scales = np.zeros((W, E // block), np.float32)
    if lib().or_qgz_reorder_quant(_p(grads), dtype, E, block, bits, N, M, _p(codes), _p(scales)):
        raise MemoryError("oracle reorder+quant failed")
    return codes, scales


def flatten_bucket(tensors, W: int):
    """A bucket given as tensors [W][n_t] -> [W][sum n_t]: rank r's bucket is row r of
    every tensor, in tensor order (the flatten that precedes the gradient exchange)."""
    return np.concatenate([np.asarray(t).reshape(W, -1) for t in tensors], axis=1)


def qgz_reorder_quant_tensors(tensors, dtype: int, block: int, bits: int, N: int, M: int):
    """Step a3 on a bucket given as tensors: flatten, then qgz_reorder_quant."""
    return qgz_reorder_quant(flatten_bucket(tensors, N * M), dtype, block, bits, N, M)


def dequant_reduce_requant(codes, scales, E: int, block: int, bits: int, N: int, M: int):
    """Hop 1: -> (codes1 uint8 [W][code_bytes(N*S)], scales1 float32 [W][N*S/block])."""
    W = N * M
    _check_topo(E, block, N, M)
    C = E // M
    codes = _contig(codes, np.uint8).reshape(W, -1)
    scales = _contig(scales, np.float32).reshape(W, -1)
    out_codes = np.zeros((W, code_bytes(C, bits)), np.uint8)
    out_scales = np.zeros((W, C // block), np.float32)
    if lib().or_dequant_reduce_requant(_p(codes), _p(scales), E, block, bits, N, M,
                                       _p(out_codes), _p(out_scales)):
        raise MemoryError("oracle dequant-reduce-requant failed")
    return out_codes, out_scales


def dequant_reduce(codes1, scales1, E: int, block: int, bits: int, N: int, M: int):
    """Hop 2: -> out float32 [W][S] (the sum over nodes)."""
    W = N * M
    _check_topo(E, block, N, M)
    S = E // W
    codes1 = _contig(codes1, np.uint8).reshape(W, -1)
    scales1 = _contig(scales1, np.float32).reshape(W, -1)
    out = np.zeros((W, S), np.float32)
    lib().or_dequant_reduce(_p(codes1), _p(scales1), E, block, bits, N, M, _p(out))
    return out


def dequant_reduce_scaled(codes1, scales1, E: int, block: int, bits: int, N: int, M: int,
                          post_scale: float, out_dtype: int = F32):
    """Hop 2 with the result multiplied by post_scale (1/W averages) and stored as
    out_dtype: -> [W][S] (float32, or uint16 bits for fp16 / bf16)."""
    W = N * M
    _check_topo(E, block, N, M)
    S = E // W
    codes1 = _contig(codes1, np.uint8).reshape(W, -1)
    scales1 = _contig(scales1, np.float32).reshape(W, -1)
    out = np.zeros((W, S), _value_dtype(out_dtype))
    if lib().or_dequant_reduce_scaled(_p(codes1), _p(scales1), E, block, bits, N, M,
                                      float(post_scale), _p(out), out_dtype):
        raise MemoryError("oracle scaled dequant-reduce failed")
    return out


def _chunks(codes, scales, length, block, bits):
    if length % block:
        raise ValueError("chunk length must be a multiple of the block")
    codes = _contig(codes, np.uint8).reshape(-1, code_bytes(length, bits))
    scales = _contig(scales, np.float32).reshape(codes.shape[0], length // block)
    return codes, scales


def dequant_reduce_requant_chunks(codes, scales, length: int, block: int, bits: int):
    """One receiver's hop 1 on the K chunks it was sent (codes [K][code_bytes(length)],
    scales [K][length/block], summed in row order) -> (codes [code_bytes(length)],
    scales [length/block])."""
    codes, scales = _chunks(codes, scales, length, block, bits)
    oc = np.zeros(code_bytes(length, bits), np.uint8)
    os_ = np.zeros(length // block, np.float32)
    if lib().or_dequant_reduce_requant_chunks(_p(codes), _p(scales), length, block, bits,
                                              codes.shape[0], _p(oc), _p(os_)):
        raise MemoryError("oracle chunk requantisation failed")
    return oc, os_


def dequant_reduce_chunks(codes, scales, length: int, block: int, bits: int,
                          post_scale: float = 1.0, out_dtype: int = F32):
    """One receiver's hop 2 on the K slices it was sent -> [length] of out_dtype holding
    fp32(sum * post_scale) (float32, or uint16 bits for fp16 / bf16)."""
    codes, scales = _chunks(codes, scales, length, block, bits)
    out = np.zeros(length, _value_dtype(out_dtype))
    lib().or_dequant_reduce_chunks(_p(codes), _p(scales), length, block, bits, codes.shape[0],
                                   float(post_scale), _p(out), out_dtype)
    return out


def qgz_passthrough(x, N: int, M: int, reorder: bool = True):
    """The two hops in plain fp32 with no quantisation: x [W][E] -> out [W][S]."""
    W = N * M
    x = _contig(x, np.float32).reshape(W, -1)
    E = x.shape[1]
    if E % W:
        raise ValueError("E must be a multiple of W")
    out = np.zeros((W, E // W), np.float32)
    if lib().or_qgz_passthrough(_p(x), E, N, M, int(bool(reorder)), _p(out)):
        raise MemoryError("oracle passthrough failed")
    return out


def qgz_pipeline(grads, dtype: int, block: int, bits: int, N: int, M: int):
    """Steps a3 -> a5 -> a7 chained; returns every intermediate."""
    W = N * M
    E = np.asarray(grads).reshape(W, -1).shape[1]
    c0, s0 = qgz_reorder_quant(grads, dtype, block, bits, N, M)
    c1, s1 = dequant_reduce_requant(c0, s0, E, block, bits, N, M)
    out = dequant_reduce(c1, s1, E, block, bits, N, M)
    return c0, s0, c1, s1, out
