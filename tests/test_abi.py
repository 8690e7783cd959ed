"""Host-side checks of the C ABI: the library loads, exports every declared symbol, the
size helpers are right, and every invalid argument is rejected on the host before any
launch (these run without a GPU; the fake addresses below never reach a kernel because
each case fails a check that precedes the launch)."""
import ctypes

import pytest
import torch

from quantized_zero_communication_gb300 import binding as zb

cpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                              reason="fake-address cases run only where no GPU exists")

FAKE = 0x10000  # 64 KiB: 32-byte aligned, never dereferenced


def test_library_exports_every_declared_symbol():
    names = zb.declared_symbols()
    assert {"zpp_quant_blockwise", "zpp_dequant_blockwise", "zpp_qgz_reorder_quant",
            "zpp_dequant_reduce_requant", "zpp_dequant_reduce", "zpp_dequant_reduce_scaled"} <= set(names)
    L = zb.lib()
    for name in names:
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_header_constants_match_binding():
    text = open(zb.HEADER).read()
    for name, val in (("ZPP_OK", 0), ("ZPP_ERR_INVALID_ARG", 1), ("ZPP_ERR_MISALIGNED", 2),
                      ("ZPP_ERR_UNSUPPORTED", 3), ("ZPP_ERR_CUDA", 4), ("ZPP_F16", 0),
                      ("ZPP_BF16", 1), ("ZPP_F32", 2)):
        assert f"{name} = {val}" in text
        assert getattr(zb, name) == val


def test_size_helpers():
    assert zb.zpp_code_bytes(1 << 20, 8) == 1 << 20
    assert zb.zpp_code_bytes(1 << 20, 4) == 1 << 19
    assert zb.zpp_code_bytes(7, 4) == 4
    assert zb.zpp_code_bytes(0, 4) == 0
    assert zb.zpp_code_bytes(5, 3) == -1
    assert zb.zpp_num_scales(1000, 256) == 4
    assert zb.zpp_num_scales(1024, 256) == 4
    assert zb.zpp_num_scales(0, 256) == 0
    # INT8 halves and INT4 quarters the fp16 bytes (4x less cross-node volume overall)
    n = 805_306_368
    assert zb.zpp_code_bytes(n, 8) * 2 == 2 * n and zb.zpp_code_bytes(n, 4) * 4 == 2 * n


def test_status_strings():
    for s in range(5):
        assert zb.zpp_status_string(s).startswith(
            ["ZPP_OK", "ZPP_ERR_INVALID_ARG", "ZPP_ERR_MISALIGNED", "ZPP_ERR_UNSUPPORTED",
             "ZPP_ERR_CUDA"][s])
    assert zb.zpp_status_string(99) == "unknown zpp_status"


@cpu_only
@pytest.mark.parametrize("bits,block,status", [
    (5, 256, zb.ZPP_ERR_INVALID_ARG), (8, 100, zb.ZPP_ERR_INVALID_ARG),
    (8, 32, zb.ZPP_ERR_INVALID_ARG), (8, 8192, zb.ZPP_ERR_INVALID_ARG),
    (4, 0, zb.ZPP_ERR_INVALID_ARG)])
def test_quant_rejects_bad_bits_and_blocks(bits, block, status):
    assert zb.zpp_quant_blockwise(FAKE, zb.ZPP_F16, 4096, block, bits, FAKE, FAKE) == status
    assert zb.zpp_dequant_blockwise(FAKE, FAKE, 4096, block, bits, FAKE, zb.ZPP_F16) == status


@cpu_only
def test_quant_rejects_bad_pointers_sizes_and_types():
    q, d = zb.zpp_quant_blockwise, zb.zpp_dequant_blockwise
    assert q(FAKE, zb.ZPP_F16, 0, 256, 8, FAKE, FAKE) == zb.ZPP_OK         # n == 0: no-op
    assert q(0, zb.ZPP_F16, 0, 256, 8, 0, 0) == zb.ZPP_OK
    assert q(FAKE, zb.ZPP_F16, -1, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_INVALID_ARG
    assert q(FAKE, zb.ZPP_F16, (1 << 38) + 1, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_INVALID_ARG
    assert q(0, zb.ZPP_F16, 64, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_INVALID_ARG
    assert q(FAKE, zb.ZPP_F16, 64, 256, 8, 0, FAKE) == zb.ZPP_ERR_INVALID_ARG
    assert q(FAKE, zb.ZPP_F16, 64, 256, 8, FAKE, 0) == zb.ZPP_ERR_INVALID_ARG
    assert q(FAKE, 7, 64, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_INVALID_ARG
    assert q(FAKE, zb.ZPP_F32, 64, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_UNSUPPORTED
    assert q(FAKE + 8, zb.ZPP_F16, 64, 256, 8, FAKE, FAKE) == zb.ZPP_ERR_MISALIGNED
    assert q(FAKE, zb.ZPP_BF16, 64, 256, 8, FAKE + 8, FAKE) == zb.ZPP_ERR_MISALIGNED
    assert q(FAKE, zb.ZPP_BF16, 64, 256, 8, FAKE, FAKE + 2) == zb.ZPP_ERR_MISALIGNED
    assert d(FAKE, FAKE, 64, 256, 8, FAKE, 9) == zb.ZPP_ERR_INVALID_ARG
    assert d(FAKE + 8, FAKE, 64, 256, 8, FAKE, zb.ZPP_F16) == zb.ZPP_ERR_MISALIGNED
    assert d(FAKE, FAKE, 64, 256, 8, FAKE + 8, zb.ZPP_F32) == zb.ZPP_ERR_MISALIGNED
    assert d(FAKE, FAKE + 1, 64, 256, 8, FAKE, zb.ZPP_F32) == zb.ZPP_ERR_MISALIGNED
    assert d(FAKE, FAKE, 0, 256, 8, FAKE, zb.ZPP_F16) == zb.ZPP_OK


@cpu_only
def test_qgz_entry_points_reject_bad_topologies():
    T = zb.Topology
    fns = [
        lambda E, B, b, t, p=FAKE: zb.zpp_qgz_reorder_quant(p, zb.ZPP_BF16, E, B, b, t, FAKE, FAKE),
        lambda E, B, b, t, p=FAKE: zb.zpp_dequant_reduce_requant(p, FAKE, E, B, b, t, FAKE, FAKE),
        lambda E, B, b, t, p=FAKE: zb.zpp_dequant_reduce(p, FAKE, E, B, b, t, FAKE),
    ]
    for f in fns:
        assert f(8 * 128, 128, 4, T(0, 4)) == zb.ZPP_ERR_INVALID_ARG     # N < 1
        assert f(8 * 128, 128, 4, T(2, 0)) == zb.ZPP_ERR_INVALID_ARG     # M < 1
        assert f(65536 * 64, 64, 4, T(256, 256)) == zb.ZPP_ERR_INVALID_ARG  # W > 65535
        assert f(8 * 128 + 128, 128, 4, T(2, 4)) == zb.ZPP_ERR_INVALID_ARG  # E % (W*B)
        assert f(8 * 128, 128, 6, T(2, 4)) == zb.ZPP_ERR_INVALID_ARG     # bits
        assert f(8 * 96, 96, 4, T(2, 4)) == zb.ZPP_ERR_INVALID_ARG       # block not 2^k
        assert f(1 << 31, 128, 4, T(2, 4)) == zb.ZPP_ERR_INVALID_ARG     # E >= 2^31
        assert f(-8 * 128, 128, 4, T(2, 4)) == zb.ZPP_ERR_INVALID_ARG
        assert f(0, 128, 4, T(2, 4)) == zb.ZPP_OK                        # empty: no-op
        assert f(8 * 128, 128, 4, T(2, 4), 0) == zb.ZPP_ERR_INVALID_ARG  # null input
        assert f(8 * 128, 128, 4, T(2, 4), FAKE + 8) == zb.ZPP_ERR_MISALIGNED
    assert zb.zpp_qgz_reorder_quant(FAKE, zb.ZPP_F32, 1024, 128, 4, T(2, 4), FAKE,
                                    FAKE) == zb.ZPP_ERR_UNSUPPORTED
    R = zb.LocalRange
    for lr, want in (((0, 4), zb.ZPP_OK), ((2, 2), zb.ZPP_OK), ((-1, 2), zb.ZPP_ERR_INVALID_ARG),
                     ((3, 2), zb.ZPP_ERR_INVALID_ARG), ((0, 5), zb.ZPP_ERR_INVALID_ARG)):
        rng = R(*lr)
        if want == zb.ZPP_OK and lr[0] != lr[1]:
            continue  # a non-empty valid range would launch: not on fake addresses
        assert zb.zpp_qgz_reorder_quant_range(FAKE, zb.ZPP_BF16, 1024, 128, 4, T(2, 4), rng,
                                              FAKE, FAKE) == want
        assert zb.zpp_dequant_reduce_requant_range(FAKE, FAKE, 1024, 128, 4, T(2, 4), rng, FAKE,
                                                   FAKE) == want
        assert zb.zpp_dequant_reduce_scaled_range(FAKE, FAKE, 1024, 128, 4, T(2, 4), rng, 1.0,
                                                  FAKE, 2) == want
    sc = zb.zpp_dequant_reduce_scaled
    assert sc(FAKE, FAKE, 1024, 128, 4, T(2, 4), 0.125, FAKE, 5) == zb.ZPP_ERR_INVALID_ARG
    assert sc(FAKE, FAKE, 1024, 128, 4, T(2, 4), float("nan"), FAKE, 2) == zb.ZPP_ERR_INVALID_ARG
    assert sc(FAKE, FAKE, 1024, 128, 4, T(2, 4), float("inf"), FAKE, 2) == zb.ZPP_ERR_INVALID_ARG
    assert sc(FAKE, FAKE, 1024, 128, 4, T(2, 4), 0.125, FAKE + 8, 1) == zb.ZPP_ERR_MISALIGNED
    assert sc(FAKE, FAKE, 1000, 128, 4, T(2, 4), 0.125, FAKE, 1) == zb.ZPP_ERR_INVALID_ARG
    assert sc(FAKE, FAKE, 0, 128, 4, T(2, 4), 0.125, FAKE, 1) == zb.ZPP_OK


@cpu_only
@cpu_only
def test_tensor_bucket_entry_point_rejects_bad_tables():
    """zpp_qgz_reorder_quant_tensors: every rule on the tensor list is checked on the host."""
    topo = zb.Topology(2, 2)  # W = 4; block 128 -> E must be a multiple of 512

    def call(ptrs, sizes, dt=zb.ZPP_BF16, block=128, bits=4, t=topo, codes=FAKE, scales=FAKE):
        return zb.zpp_qgz_reorder_quant_tensors(ptrs, sizes, dt, block, bits, t, codes, scales)

    INV, MIS, UNS = zb.ZPP_ERR_INVALID_ARG, zb.ZPP_ERR_MISALIGNED, zb.ZPP_ERR_UNSUPPORTED
    assert zb.lib().zpp_qgz_reorder_quant_tensors(None, None, 1, zb.ZPP_BF16, 128, 4, topo,
                                                   FAKE, FAKE, None) == INV
    assert call([], []) == INV                                       # no tensor
    assert call([FAKE] * 1025, [16] * 1025) == INV                   # over ZPP_MAX_TENSORS
    assert call([FAKE, FAKE], [528, -16]) == INV                     # negative size
    assert call([FAKE, FAKE], [256, 240]) == INV                     # E % (W * block) != 0
    assert call([FAKE], [1 << 31]) == INV                            # E >= 2^31
    assert call([FAKE, FAKE], [256, 256], t=zb.Topology(0, 2)) == INV
    assert call([FAKE, FAKE], [256, 256], bits=3) == INV
    assert call([FAKE, FAKE], [256, 256], dt=7) == INV
    assert call([FAKE, 0], [256, 256]) == INV                        # null tensor
    assert call([FAKE, FAKE], [256, 256], codes=0) == INV
    assert call([FAKE, FAKE], [256, 256], dt=zb.ZPP_F32) == UNS
    assert call([FAKE, FAKE], [264, 248]) == MIS                     # not a multiple of 16
    assert call([FAKE, FAKE + 8], [256, 256]) == MIS                 # pointer not 16-byte aligned
    assert call([FAKE, FAKE], [256, 256], codes=FAKE + 8) == MIS
    assert call([FAKE, FAKE], [256, 256], scales=FAKE + 2) == MIS
    assert call([0, 0], [0, 0]) == zb.ZPP_OK                         # empty bucket: no launch


def test_fault_query_and_wait_selftest_reject_bad_arguments():
    L = zb.lib()
    assert L.zpp_device_fault(None, 0) == zb.ZPP_ERR_INVALID_ARG
    assert L.zpp_wait_selftest(0, None) == zb.ZPP_ERR_INVALID_ARG
    assert L.zpp_wait_selftest(10_000_000_001, None) == zb.ZPP_ERR_INVALID_ARG


def test_copy_rejects_bad_sizes():
    assert zb.zpp_device_copy(FAKE, FAKE * 2, 33) == zb.ZPP_ERR_INVALID_ARG
    assert zb.zpp_device_copy(FAKE, FAKE * 2, 0) == zb.ZPP_OK
    assert zb.zpp_device_copy(FAKE + 16, FAKE * 2, 64) == zb.ZPP_ERR_MISALIGNED


def test_tensor_helpers_refuse_cpu_tensors():
    x = torch.zeros(256, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        zb.quant_blockwise(x, 256, 8)
