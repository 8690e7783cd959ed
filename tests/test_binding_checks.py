"""The tensor wrappers refuse buffers that do not fit the call before anything reaches
libzpp: wrong element counts (too small or too large for n / E / W), wrong dtypes, and
layouts of the wrong hop. These run without a GPU: the size and dtype checks come before
the device check, and every case below fails one of them (the message says which)."""
import pytest
import torch

import quantized_zero_communication_gb300 as zpp
from quantized_zero_communication_gb300 import binding as zb

U8, F32, F16, BF16 = torch.uint8, torch.float32, torch.float16, torch.bfloat16


def z(n, dtype=U8):
    return torch.zeros(n, dtype=dtype)


def raises(match, fn):
    with pytest.raises(ValueError, match=match):
        fn()


def test_quant_blockwise_checks():
    x = z(1000, F16)
    raises("codes: 999 elements, expected 1000", lambda: zpp.quant_blockwise(x, 256, 8, codes=z(999)))
    raises("codes: 1000 elements, expected 500", lambda: zpp.quant_blockwise(x, 256, 4, codes=z(1000)))
    raises("scales: 3 elements, expected 4", lambda: zpp.quant_blockwise(x, 256, 8, scales=z(3, F32)))
    raises("scales: dtype", lambda: zpp.quant_blockwise(x, 256, 8, scales=z(4, torch.float64)))
    raises("codes: dtype", lambda: zpp.quant_blockwise(x, 256, 8, codes=z(1000, torch.int32)))
    raises("x: dtype", lambda: zpp.quant_blockwise(z(1000, F32), 256, 8))
    raises("CUDA tensors only", lambda: zpp.quant_blockwise(x, 256, 8, codes=z(1000), scales=z(4, F32)))


def test_dequant_blockwise_checks():
    # INT4: n larger than two codes per byte can hold
    raises("codes: 500 elements, expected 501",
           lambda: zpp.dequant_blockwise(z(500), z(4, F32), 1001, 256, 4))
    raises("scales: 3 elements, expected 4",
           lambda: zpp.dequant_blockwise(z(1000), z(3, F32), 1000, 256, 8))
    raises("y: 999 elements, expected 1000",
           lambda: zpp.dequant_blockwise(z(1000), z(4, F32), 1000, 256, 8, y=z(999, F16)))
    raises("y: dtype", lambda: zpp.dequant_blockwise(z(1000), z(4, F32), 1000, 256, 8,
                                                     y=z(1000, torch.int32)))


def test_qgz_step1_checks():
    N, M, B = 2, 2, 64
    W, E = N * M, 4 * 2 * 64
    g = z(W * E, BF16)
    raises("do not split into 4 ranks", lambda: zpp.qgz_reorder_quant(z(W * E + 1, BF16), B, 4, N, M))
    raises("codes: 511 elements, expected 1024",
           lambda: zpp.qgz_reorder_quant(g, B, 4, N, M, codes=z(511)))
    raises("scales: 15 elements, expected 32",
           lambda: zpp.qgz_reorder_quant(g, B, 4, N, M, scales=z(15, F32)))
    raises("grads: dtype", lambda: zpp.qgz_reorder_quant(z(W * E, F32), B, 4, N, M))
    raises("tensors\\[1\\]: dtype",
           lambda: zpp.qgz_reorder_quant_tensors([z(W * 256, BF16), z(W * 256, F16)], B, 4, N, M))
    raises("W equal per-rank copies",
           lambda: zpp.qgz_reorder_quant_tensors([z(W * 256 + 1, BF16)], B, 4, N, M))
    raises("codes: 3 elements", lambda: zpp.qgz_reorder_quant_tensors(
        [z(W * 256, BF16), z(W * 256, BF16)], B, 4, N, M, codes=z(3)))


def test_qgz_hop_checks():
    N, M, B, bits = 2, 2, 64, 4
    W, E = N * M, 4 * 2 * 64
    C = E // M
    c0, s0 = z(W * E // 2), z(W * E // B, F32)        # step-1 layout
    c1, s1 = z(W * C // 2), z(W * C // B, F32)        # hop-1 layout
    # hop 1 reads the step-1 layout
    raises("codes: 512 elements, expected 1024",
           lambda: zpp.dequant_reduce_requant(c1, s0, E, B, bits, N, M))
    raises("scales: 16 elements, expected 32",
           lambda: zpp.dequant_reduce_requant(c0, s1, E, B, bits, N, M))
    raises("out_codes: 1024 elements, expected 512",
           lambda: zpp.dequant_reduce_requant(c0, s0, E, B, bits, N, M, out_codes=c0))
    raises("out_scales: 32 elements, expected 16",
           lambda: zpp.dequant_reduce_requant(c0, s0, E, B, bits, N, M, out_scales=z(32, F32)))
    # an E that does not match the buffers
    raises("codes: 1024 elements, expected 2048",
           lambda: zpp.dequant_reduce_requant(c0, s0, 2 * E, B, bits, N, M))
    # hop 2 reads the hop-1 layout
    raises("codes: 1024 elements, expected 512", lambda: zpp.dequant_reduce(c0, s1, E, B, bits, N, M))
    raises("out: 511 elements, expected 512",
           lambda: zpp.dequant_reduce(c1, s1, E, B, bits, N, M, out=z(511, F32)))
    raises("out: dtype", lambda: zpp.dequant_reduce(c1, s1, E, B, bits, N, M, out=z(512, F16)))
    raises("out: dtype", lambda: zpp.dequant_reduce_scaled(c1, s1, E, B, bits, N, M,
                                                           out=z(512, torch.int32)))


def test_pipelined_and_copy_checks():
    N, M, B, bits = 2, 2, 64, 4
    W, E = N * M, 4 * 2 * 64
    g = z(W * E, BF16)
    good = dict(c0=z(W * E // 2), s0=z(W * E // B, F32), c1=z(W * E // M // 2),
                s1=z(W * E // M // B, F32), out=z(E, F32))
    bad = dict(good, c1=z(7))
    raises("bufs.c1: 7 elements", lambda: zb.qgz_pipelined(g, B, bits, N, M,
                                                           bufs=zb.QgzBuffers(**bad)))
    raises("multiple of W \\* block", lambda: zb.qgz_pipelined(z(W * 96, BF16), B, bits, N, M))
    raises("CUDA tensors only", lambda: zb.qgz_pipelined(g, B, bits, N, M,
                                                         bufs=zb.QgzBuffers(**good)))
    raises("dst holds 8 bytes, src 16", lambda: zpp.device_copy(z(16), z(8)))
