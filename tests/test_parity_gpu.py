"""GPU parity: every kernel, called through the C ABI, against the CPU oracle on the same
seeded inputs. Codes, scales, dequantised fp16/bf16 values and the reorder permutation
must match bit for bit; fp32 sums (fixed ascending order, each term added with one
rounding as a fused multiply-add) are required within 1e-6 relative and are expected to
match exactly, which is also checked.

Sizes span several warp tiles plus a ragged tail, every block size and both code widths,
the small and the full-size workloads, and the edge cases (empty, one element, odd
lengths, blocks longer than the data, the largest block)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_zero_communication_gb300 as zpp
from quantized_zero_communication_gb300 import binding as zb
from quantized_zero_communication_gb300 import inputs

pytestmark = pytest.mark.gpu

BLOCKS = (64, 128, 256, 512, 1024, 2048, 4096)
DEV = "cuda:0"
REL_TOL = 1e-6  # fp32 reductions


def bits16(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def odt(dtype):
    return {torch.float16: oracle.F16, torch.bfloat16: oracle.BF16, torch.float32: oracle.F32}[dtype]


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_f32_parity(got, want):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= REL_TOL * np.abs(want.astype(np.float64)) + 1e-30), float(err.max())
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "fp32 sums not bit-identical"


def check_quant(x, block, bits):
    codes, scales = zpp.quant_blockwise(x, block, bits)
    oc, os_ = oracle.quant_blockwise(bits16(x), odt(x.dtype), block, bits)
    assert np.array_equal(host(codes), oc)
    assert np.array_equal(host(scales).view(np.uint32), os_.view(np.uint32))
    return codes, scales, oc, os_


# ----------------------------------------------------------------------- qwZ (K1, K2)
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_quant_dequant_all_blocks(block, bits, dtype):
    n = 3 * max(block, 2048) + 5 * 16 + 7  # several warp tiles, a ragged tile, odd tail
    kind = inputs.SWEEP_KINDS[(block + bits) % 3]
    x = inputs.draw(kind, n, seed=block + bits, dtype=dtype, device=DEV)
    codes, scales, oc, os_ = check_quant(x, block, bits)
    for out_dt in (torch.float16, torch.bfloat16, torch.float32):
        y = zpp.dequant_blockwise(codes, scales, n, block, bits, out_dt)
        oy = oracle.dequant_blockwise(oc, os_, n, block, bits, odt(out_dt))
        got = host(y.view(torch.int16)).view(np.uint16) if out_dt != torch.float32 else host(y)
        assert np.array_equal(got.view(oy.dtype), oy)


@pytest.mark.parametrize("n", [1, 2, 7, 15, 16, 17, 63, 64, 65, 511, 513, 2047, 2049, 4095, 4097,
                               10_001])
@pytest.mark.parametrize("bits", [8, 4])
def test_quant_edge_lengths(n, bits):
    for block in (64, 4096):
        x = inputs.draw("uniform_outliers", n, seed=n, dtype=torch.float16, device=DEV)
        codes, scales, oc, os_ = check_quant(x, block, bits)
        y = zpp.dequant_blockwise(codes, scales, n, block, bits, torch.float16)
        oy = oracle.dequant_blockwise(oc, os_, n, block, bits, oracle.F16)
        assert np.array_equal(bits16(y), oy)


def test_golden_cases_on_gpu():
    """The hand-derived fixtures use 4-element blocks, below the ABI's minimum block of 64;
    each fixture block is embedded at the start of its own 64-element block padded with
    zeros, which leaves its absmax, scale and codes unchanged."""
    from tests.golden import load_quant_cases
    for case in load_quant_cases():
        dt = torch.float16 if case["dtype"] == "f16" else torch.bfloat16
        B, bits, n = case["block"], case["bits"], len(case["x"])
        x = torch.tensor(case["x"], dtype=torch.float64).to(dt)
        nb = -(-n // B)
        padded = torch.zeros(nb * 64, dtype=dt)
        for b in range(nb):
            seg = x[b * B:(b + 1) * B]
            padded[b * 64:b * 64 + seg.numel()] = seg
        codes, scales = zpp.quant_blockwise(padded.to(DEV), 64, bits)
        y = zpp.dequant_blockwise(codes, scales, nb * 64, 64, bits, dt)
        c, yb = host(codes), bits16(y)
        per = 64 * bits // 8
        lens = [min(B, n - b * B) for b in range(nb)]
        got = np.concatenate([c[b * per:b * per + (lens[b] * bits + 7) // 8] for b in range(nb)])
        assert list(got) == case["packed"], case["name"]
        assert list(host(scales).view(np.uint32)) == case["scale_bits"], case["name"]
        got_y = np.concatenate([yb[b * 64:b * 64 + lens[b]] for b in range(nb)])
        want_y = bits16(torch.tensor(case["y"], dtype=torch.float64).to(dt))
        assert np.array_equal(got_y, want_y), case["name"]


def test_zero_length_is_a_noop():
    x = torch.zeros(0, dtype=torch.float16, device=DEV)
    codes = torch.full((32,), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((8,), 3.0, device=DEV)
    assert zb.zpp_quant_blockwise(0, zb.ZPP_F16, 0, 256, 8,
                                  codes.data_ptr(), scales.data_ptr()) == zb.ZPP_OK
    assert torch.all(codes == 0xAB) and torch.all(scales == 3.0)


def test_invalid_arguments_write_nothing():
    x = inputs.draw("normal", 4096, seed=1, dtype=torch.float16, device=DEV)
    buf = torch.full((8192,), 0x5A, dtype=torch.uint8, device=DEV)
    sc = torch.full((64,), -1.0, device=DEV)
    st = zb.zpp_quant_blockwise(x.data_ptr() + 8, zb.ZPP_F16, 1024, 256, 8, buf.data_ptr(),
                                sc.data_ptr())
    assert st == zb.ZPP_ERR_MISALIGNED
    st = zb.zpp_quant_blockwise(x.data_ptr(), zb.ZPP_F16, 4096, 96, 8, buf.data_ptr(), sc.data_ptr())
    assert st == zb.ZPP_ERR_INVALID_ARG
    st = zb.zpp_quant_blockwise(x.data_ptr(), zb.ZPP_F16, 4096, 256, 8, buf.data_ptr() + 8,
                                sc.data_ptr())
    assert st == zb.ZPP_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.all(buf == 0x5A) and torch.all(sc == -1.0)


def at16(shape, dtype):
    """An uninitialised contiguous tensor whose data starts 16 bytes past a 32-byte boundary
    (16-byte aligned, not 32-byte aligned)."""
    n = int(np.prod(shape))
    es = torch.empty(0, dtype=dtype).element_size()
    buf = torch.empty(n + 32 // es, dtype=dtype, device=DEV)
    k = ((16 - buf.data_ptr() % 32) % 32) // es
    v = buf[k:k + n].view(shape)
    assert v.data_ptr() % 32 == 16
    return v


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("bits", [8, 4])
def test_sixteen_byte_aligned_buffers_are_served(dtype, bits):
    """Every entry point on buffers that are 16-byte but not 32-byte aligned (fp16 / bf16
    input at an 8-element offset) takes its 128-bit path and gives the oracle's bits."""
    n, B = 3 * 4096 + 512, 256
    x = at16((n,), dtype)
    x.copy_(inputs.draw("normal", n, seed=3 + bits, dtype=dtype, device=DEV))
    codes = at16((zb.zpp_code_bytes(n, bits),), torch.uint8)
    scales = at16((zb.zpp_num_scales(n, B),), torch.float32)
    zpp.quant_blockwise(x, B, bits, codes, scales)
    oc, os_ = oracle.quant_blockwise(bits16(x), odt(dtype), B, bits)
    assert np.array_equal(host(codes), oc)
    assert np.array_equal(host(scales).view(np.uint32), os_.view(np.uint32))
    for ydt in (torch.float16, torch.bfloat16, torch.float32):
        y = zpp.dequant_blockwise(codes, scales, n, B, bits, y=at16((n,), ydt))
        oy = oracle.dequant_blockwise(oc, os_, n, B, bits, odt(ydt))
        assert np.array_equal(host(y.view(torch.uint8)), oy.view(np.uint8))

    N, M = 2, 4
    W, C = N * M, None
    E = W * (2 * 8192 + 512)
    C = E // M
    g = at16((W, E), dtype)
    g.copy_(inputs.draw("laplace", W * E, seed=9 + bits, dtype=dtype, device=DEV).reshape(W, E))
    c0 = at16((W, zb.zpp_code_bytes(E, bits)), torch.uint8)
    s0 = at16((W, E // B), torch.float32)
    zpp.qgz_reorder_quant(g, B, bits, N, M, codes=c0, scales=s0)
    c1 = at16((W, zb.zpp_code_bytes(C, bits)), torch.uint8)
    s1 = at16((W, C // B), torch.float32)
    zpp.dequant_reduce_requant(c0, s0, E, B, bits, N, M, out_codes=c1, out_scales=s1)
    out = zpp.dequant_reduce(c1, s1, E, B, bits, N, M, out=at16((W, E // W), torch.float32))
    avg = zpp.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, post_scale=1.0 / W,
                                    out=at16((W, E // W), dtype))
    want = oracle.qgz_pipeline(bits16(g).reshape(W, E), odt(dtype), B, bits, N, M)
    for a, b, name in zip((c0, s0, c1, s1), want[:4], ("codes", "scales", "hop-1 codes",
                                                      "hop-1 scales")):
        assert np.array_equal(host(a).view(np.uint8), b.view(np.uint8)), name
    assert_f32_parity(host(out), want[4])
    wavg = oracle.dequant_reduce_scaled(want[2], want[3], E, B, bits, N, M, 1.0 / W, odt(dtype))
    assert np.array_equal(bits16(avg).reshape(-1), np.asarray(wavg).reshape(-1).view(np.uint16))

    sizes = inputs.random_sizes(E, 5, seed=bits)
    tensors = []
    for t in inputs.split_bucket(g, sizes):
        v = at16(tuple(t.shape), dtype)
        v.copy_(t)
        tensors.append(v)
    tc, ts = zpp.qgz_reorder_quant_tensors(tensors, B, bits, N, M)
    assert torch.equal(tc, c0) and torch.equal(ts.view(torch.int32), s0.view(torch.int32))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,M", [(3, 2), (2, 1)])
def test_sixteen_byte_aligned_small_hops(N, M, bits):
    """The fused hop with one or two sources on codes that are 16-byte but not 32-byte
    aligned (INT8: the wide kernel's 128-bit loads and stores; INT4: the kernel that loads
    two tiles ahead), over whole tiles and a ragged last tile."""
    B = 256
    W = N * M
    E = W * (2 * 8192 + 512)
    C = E // M
    g = inputs.draw("laplace", W * E, seed=21 + bits + M, dtype=torch.bfloat16,
                    device=DEV).reshape(W, E)
    c0 = at16((W, zb.zpp_code_bytes(E, bits)), torch.uint8)
    s0 = at16((W, E // B), torch.float32)
    zpp.qgz_reorder_quant(g, B, bits, N, M, codes=c0, scales=s0)
    c1 = at16((W, zb.zpp_code_bytes(C, bits)), torch.uint8)
    s1 = at16((W, C // B), torch.float32)
    zpp.dequant_reduce_requant(c0, s0, E, B, bits, N, M, out_codes=c1, out_scales=s1)
    want = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    for a, b, name in zip((c0, s0, c1, s1), want[:4], ("codes", "scales", "hop-1 codes",
                                                      "hop-1 scales")):
        assert np.array_equal(host(a).view(np.uint8), b.view(np.uint8)), name


def test_shard_launches_equal_one_launch():
    """qwZ quantises per rank; 16 shard launches at their offsets == one launch."""
    n_shard, R, B = 2048 * 24, 16, 2048
    x = inputs.draw("normal", n_shard * R, seed=77, dtype=torch.float16, device=DEV)
    c_all, s_all = zpp.quant_blockwise(x, B, 8)
    c_sh = torch.empty_like(c_all)
    s_sh = torch.empty_like(s_all)
    for r in range(R):
        zpp.quant_blockwise(x[r * n_shard:(r + 1) * n_shard], B, 8,
                            codes=c_sh[r * n_shard:(r + 1) * n_shard],
                            scales=s_sh[r * n_shard // B:(r + 1) * n_shard // B])
    torch.cuda.synchronize()
    assert torch.equal(c_all, c_sh) and torch.equal(s_all, s_sh)


def test_repeat_calls_are_deterministic():
    x = inputs.draw("laplace", 1 << 20, seed=3, dtype=torch.bfloat16, device=DEV)
    a = zpp.quant_blockwise(x, 512, 4)
    b = zpp.quant_blockwise(x, 512, 4)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_qwz_round_trip_workload():
    x = inputs.qwz_round_trip(DEV)
    codes, scales, oc, os_ = check_quant(x, 256, 8)
    y = zpp.dequant_blockwise(codes, scales, x.numel(), 256, 8, torch.float16)
    assert np.array_equal(bits16(y), oracle.dequant_blockwise(oc, os_, x.numel(), 256, 8, oracle.F16))


# ----------------------------------------------------------------------- qgZ (K3, K4, K5)
TOPOS = [(1, 1), (1, 2), (2, 1), (2, 2), (2, 4), (3, 2), (4, 3), (2, 6), (1, 8), (1, 12), (1, 16),
         (2, 16), (1, 32), (8, 2), (16, 1), (4, 8)]


def run_qgz(g, block, bits, N, M):
    E = g.shape[1]
    c0, s0 = zpp.qgz_reorder_quant(g, block, bits, N, M)
    c1, s1 = zpp.dequant_reduce_requant(c0, s0, E, block, bits, N, M)
    out = zpp.dequant_reduce(c1, s1, E, block, bits, N, M)
    res = [host(t) for t in (c0, s0, c1, s1, out)]
    # no bounded wait of the INT8 fused hop ran out
    assert zb.zpp_device_fault() == 0
    return res


def check_qgz(g, block, bits, N, M):
    got = run_qgz(g, block, bits, N, M)
    want = oracle.qgz_pipeline(bits16(g), odt(g.dtype), block, bits, N, M)
    names = ("reordered codes", "source scales", "hop-1 codes", "hop-1 scales")
    for a, b, name in zip(got[:4], want[:4], names):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name
    assert_f32_parity(got[4], want[4])


@pytest.mark.parametrize("N,M", TOPOS)
@pytest.mark.parametrize("bits", [4, 8])
def test_qgz_pipeline_topologies(N, M, bits):
    W = N * M
    for block in (64, 512, 4096):
        # a slice of two blocks plus one slice spanning several tiles
        for per_slice in (2 * block, 3 * 8192 + block):
            if W * W * per_slice > (1 << 24):
                continue
            E = W * per_slice
            g = inputs.draw("laplace", W * E, seed=W + block, dtype=torch.bfloat16,
                            device=DEV).reshape(W, E)
            check_qgz(g, block, bits, N, M)


def test_bounded_wait_reports_and_the_context_stays_usable():
    """A wait that nothing completes ends after its limit and sets its fault bit; the
    device keeps working afterwards (an INT8 exchange then matches the oracle and leaves
    the fault word clear)."""
    zb.zpp_device_fault(clear=True)
    assert zb.zpp_wait_selftest(20_000_000, torch.cuda.current_stream().cuda_stream) == zb.ZPP_OK
    torch.cuda.synchronize()
    assert zb.zpp_device_fault(clear=True) == 4
    assert zb.zpp_device_fault() == 0
    g = inputs.draw("laplace", 8 * 8 * 4096, seed=5, dtype=torch.bfloat16,
                    device=DEV).reshape(8, 8 * 4096)
    check_qgz(g, 256, 8, 2, 4)


# ----------------------------------------------------------------------- fused bucket flatten
def check_tensor_bucket(g, sizes, block, bits, N, M):
    """K3 over `g` cut into tensors of `sizes` == the oracle on the flattened tensors == the
    flat-buffer K3 on `g` (all bit for bit)."""
    tensors = inputs.split_bucket(g, sizes)
    c, s = zpp.qgz_reorder_quant_tensors(tensors, block, bits, N, M)
    oc, os_ = oracle.qgz_reorder_quant_tensors([bits16(t).reshape(t.shape) for t in tensors],
                                               odt(g.dtype), block, bits, N, M)
    assert np.array_equal(host(c), oc)
    assert np.array_equal(host(s).view(np.uint32), os_.view(np.uint32))
    fc, fs = zpp.qgz_reorder_quant(g, block, bits, N, M)
    assert torch.equal(c, fc) and torch.equal(s.view(torch.int32), fs.view(torch.int32))


@pytest.mark.parametrize("N,M", [(1, 1), (2, 2), (2, 4), (3, 2), (4, 8)])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_tensor_bucket_equals_flattened_bucket(N, M, bits, dtype):
    """Tensors of seeded random sizes (multiples of 16, empty ones included) whose edges
    fall inside blocks, tiles and slices; 1, 5 and 17 tensors."""
    W = N * M
    for block, count in ((64, 1), (512, 5), (4096, 17)):
        per_slice = 3 * 8192 + block if W * W * (3 * 8192 + block) <= (1 << 24) else 2 * block
        E = W * per_slice
        g = inputs.draw("laplace", W * E, seed=31 * W + block + bits, dtype=dtype,
                        device=DEV).reshape(W, E)
        sizes = inputs.random_sizes(E, count, seed=W + count)
        check_tensor_bucket(g, sizes, block, bits, N, M)


def test_tensor_bucket_largest_table():
    """ZPP_MAX_TENSORS tensors, many of them one 16-element vector per rank; one more is
    refused on the host."""
    N, M, block = 2, 2, 64
    W = N * M
    E = W * block * 64  # 16384 elements per rank
    g = inputs.draw("normal", W * E, seed=77, dtype=torch.bfloat16, device=DEV).reshape(W, E)
    sizes = inputs.random_sizes(E, 1024, seed=78)
    check_tensor_bucket(g, sizes, block, 4, N, M)
    tensors = inputs.split_bucket(g, [16] * 1023 + [E - 16 * 1023 - 16, 16])
    with pytest.raises(zb.ZppError):
        zpp.qgz_reorder_quant_tensors(tensors, block, 4, N, M)


def test_tensor_bucket_rejects_unaligned_sizes():
    g = torch.zeros((4, 1024), dtype=torch.float16, device=DEV)
    with pytest.raises(zb.ZppError) as e:
        zpp.qgz_reorder_quant_tensors(inputs.split_bucket(g, [24, 1000]), 64, 4, 2, 2)
    assert e.value.status == zb.ZPP_ERR_MISALIGNED


@pytest.mark.parametrize("N,M", [(2, 4), (3, 2), (4, 8)])
@pytest.mark.parametrize("bits", [4, 8])
def test_averaged_owner_slices(N, M, bits):
    """zpp_dequant_reduce_scaled: 1/W (and an arbitrary scale) into fp32, bf16 and fp16."""
    W, B = N * M, 256
    E = W * 2 * 4096
    g = inputs.draw("laplace", W * E, seed=W * bits, dtype=torch.bfloat16, device=DEV).reshape(W, E)
    c0, s0 = zpp.qgz_reorder_quant(g, B, bits, N, M)
    c1, s1 = zpp.dequant_reduce_requant(c0, s0, E, B, bits, N, M)
    oc1, os1 = host(c1), host(s1)
    plain = zpp.dequant_reduce(c1, s1, E, B, bits, N, M)
    for ps in (1.0 / W, 0.3, 1.0):
        for dt in (torch.float32, torch.bfloat16, torch.float16):
            got = zpp.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, post_scale=ps, dtype=dt)
            want = oracle.dequant_reduce_scaled(oc1, os1, E, B, bits, N, M, ps, odt(dt))
            if dt == torch.float32:
                assert_f32_parity(host(got), want)
            else:
                assert np.array_equal(bits16(got), want)
    one = zpp.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, post_scale=1.0)
    torch.cuda.synchronize()
    assert torch.equal(one, plain)


@pytest.mark.parametrize("N,M", [(2, 4), (3, 2), (1, 8), (4, 8)])
@pytest.mark.parametrize("n_streams", [1, 2, 3])
def test_pipelined_subexchanges_equal_the_whole(N, M, n_streams):
    """The local-index sub-pipelines on several streams give the same buffers, bit for bit,
    as the three unrestricted calls."""
    W, B, bits = N * M, 512, 4
    E = W * 2 * 4096
    g = inputs.draw("laplace", W * E, seed=31 * W + n_streams, dtype=torch.bfloat16,
                    device=DEV).reshape(W, E)
    bufs = zpp.qgz_pipelined(g, B, bits, N, M, n_streams=n_streams)
    whole = run_qgz(g, B, bits, N, M)
    split = zpp.qgz_pipelined(g, B, bits, N, M, chunks=n_streams, streams=(
        "split", torch.cuda.Stream(DEV), torch.cuda.Stream(DEV, priority=-1)))
    for a, b in zip([host(t) for t in (split.c0, split.s0, split.c1, split.s1, split.out)], whole):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    got = [host(t) for t in (bufs.c0, bufs.s0, bufs.c1, bufs.s1, bufs.out)]
    for a, b in zip(got, whole):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_qgz_fp16_gradients():
    g = inputs.draw("normal", 8 * 8 * 1024, seed=4, dtype=torch.float16, device=DEV).reshape(8, -1)
    check_qgz(g, 128, 4, 2, 4)


def test_golden_qgz_fused_sum_on_gpu():
    from tests.golden import load_qgz_case
    from tests.test_oracle_pins import check_qgz_case, qgz_case_inputs
    case = load_qgz_case()
    g = qgz_case_inputs(case).to(DEV)
    got = run_qgz(g, case["block"], case["bits"], case["N"], case["M"])
    check_qgz_case(case, *got)


def test_qgz_tiny_workload():
    check_qgz(inputs.qgz_tiny(DEV), 128, 4, 2, 4)


@pytest.mark.parametrize("K", [2, 8, 16])
@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_reduce_requant_sweep_shapes(K, bits):
    """The sweep's K-way fused reduction: topology {1 node, K GPUs}."""
    for block in (64, 256, 1024, 4096):
        E = K * block * 4
        g = inputs.draw("uniform_outliers", K * E, seed=K * block, dtype=torch.float16,
                        device=DEV).reshape(K, E)
        check_qgz(g, block, bits, 1, K)


# ----------------------------------------------------------------------- the sweep
SWEEP_16M = [r for r in inputs.sweep_rows() if r["size"] == 1 << 24]


@pytest.mark.parametrize("row", SWEEP_16M, ids=lambda r: f"{str(r['dtype'])[6:]}-int{r['bits']}-B{r['block']}-{r['kind']}")
def test_sweep_rows_quant_dequant(row):
    """Every sweep row (dtype x bits x block x distribution) at 2^24 elements, its own seed."""
    x = inputs.draw(row["kind"], row["size"], seed=row["seed"], dtype=row["dtype"], device=DEV)
    codes, scales, oc, os_ = check_quant(x, row["block"], row["bits"])
    y = zpp.dequant_blockwise(codes, scales, x.numel(), row["block"], row["bits"], row["dtype"])
    oy = oracle.dequant_blockwise(oc, os_, x.numel(), row["block"], row["bits"], odt(row["dtype"]))
    assert np.array_equal(bits16(y), oy)


@pytest.mark.parametrize("K", [2, 8, 16])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", inputs.SWEEP_BLOCKS)
def test_sweep_fused_reduction(K, bits, block):
    """The sweep's fused dequant-reduce-requant with K in {2, 8, 16} (topology 1 x K) on
    2^24 elements in total."""
    n = 1 << 24
    g = inputs.draw("laplace", n, seed=7 * K + block + bits, dtype=torch.bfloat16,
                    device=DEV).reshape(K, n // K)
    check_qgz(g, block, bits, 1, K)


# ----------------------------------------------------------------------- full-size workloads
@pytest.mark.slow
def test_gpt_layer_full_size():
    """qwZ on one hidden-8192 GPT layer: 805,306,368 fp16 weights, INT8 block 2048,
    quantised in one launch (16 block-aligned shards) and dequantised after the gather."""
    x = inputs.gpt_layer(DEV)
    n = x.numel()
    codes, scales = zpp.quant_blockwise(x, 2048, 8)
    y = zpp.dequant_blockwise(codes, scales, n, 2048, 8, torch.float16)
    xb = bits16(x)
    oc, os_ = oracle.quant_blockwise(xb, oracle.F16, 2048, 8)
    assert np.array_equal(host(codes), oc)
    assert np.array_equal(host(scales).view(np.uint32), os_.view(np.uint32))
    del codes
    oy = oracle.dequant_blockwise(oc, os_, n, 2048, 8, oracle.F16)
    assert np.array_equal(bits16(y), oy)


@pytest.mark.slow
def test_gradient_bucket_full_size():
    """qgZ on a 536,870,912-element bf16 bucket over 4 nodes x 8 GPUs, INT4 block 512."""
    g = inputs.gradient_bucket(DEV)
    check_qgz(g, 512, 4, 4, 8)


@pytest.mark.slow
def test_gradient_bucket_as_tensors_full_size():
    """The 4 x 8 bucket given as its 13 parameter-gradient tensors per rank: the fused
    flatten equals the oracle on the flattened bucket and the flat-buffer K3."""
    g = inputs.gradient_bucket(DEV)
    check_tensor_bucket(g, inputs.bucket_tensor_sizes(), 512, 4, 4, 8)


@pytest.mark.slow
@pytest.mark.parametrize("bits", [8, 4])
def test_largest_sweep_size(bits):
    """The sweep's largest size (2^30 elements) through quant, dequant and the fused
    K-way reduction, checked against the oracle on the whole tensor."""
    n = 1 << 30
    x = inputs.draw("uniform_outliers", n, seed=999, dtype=torch.bfloat16, device=DEV)
    codes, scales, oc, os_ = check_quant(x, 4096, bits)
    y = zpp.dequant_blockwise(codes, scales, n, 4096, bits, torch.bfloat16)
    assert np.array_equal(bits16(y), oracle.dequant_blockwise(oc, os_, n, 4096, bits, oracle.BF16))
    del x, y, codes, scales
    K = 16
    g = inputs.draw("normal", n, seed=1000, dtype=torch.bfloat16, device=DEV).reshape(K, n // K)
    E = n // K
    c0, s0 = zpp.qgz_reorder_quant(g, 1024, bits, 1, K)
    c1, s1 = zpp.dequant_reduce_requant(c0, s0, E, 1024, bits, 1, K)
    oc0, os0 = oracle.qgz_reorder_quant(bits16(g), oracle.BF16, 1024, bits, 1, K)
    assert np.array_equal(host(c0), oc0)
    oc1, os1 = oracle.dequant_reduce_requant(oc0, os0, E, 1024, bits, 1, K)
    assert np.array_equal(host(c1), oc1)
    assert np.array_equal(host(s1).view(np.uint32), os1.view(np.uint32))


@pytest.mark.slow
def test_offsets_beyond_2_pow_31():
    """n = 2^31 + 2^20 + 77 fp16 elements (4.3 GB): quant and dequant through 64-bit offsets.
    Quantisation is block-local, so the oracle checks windows of whole blocks one by one:
    the start, both sides of element 2^31, and the ragged tail."""
    n, B = (1 << 31) + (1 << 20) + 77, 1024
    x = torch.empty(n, dtype=torch.float16, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(2024)
    for i in range(0, n, 1 << 28):  # draw in pieces to bound the fp32 temporary
        m = min(1 << 28, n - i)
        x[i:i + m] = (torch.randn(m, generator=g, device=DEV) * 0.02).half()
    codes, scales = zpp.quant_blockwise(x, B, 8)
    y = zpp.dequant_blockwise(codes, scales, n, B, 8, torch.float16)
    torch.cuda.synchronize()
    for lo in (0, (1 << 31) - 64 * B, n - (n % B) - 64 * B):
        hi = min(n, lo + 128 * B)
        xb = bits16(x[lo:hi])
        oc, os_ = oracle.quant_blockwise(xb, oracle.F16, B, 8)
        assert np.array_equal(codes[lo:hi].cpu().numpy(), oc), lo
        assert np.array_equal(scales[lo // B:(hi + B - 1) // B].cpu().numpy().view(np.uint32),
                              os_.view(np.uint32)), lo
        assert np.array_equal(bits16(y[lo:hi]), oracle.dequant_blockwise(oc, os_, hi - lo, B, 8,
                                                                         oracle.F16)), lo


def test_device_copy():
    a = torch.randint(0, 255, (1 << 20,), dtype=torch.uint8, device=DEV)
    b = torch.zeros_like(a)
    zpp.device_copy(a, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ----------------------------------------------------------------------- one real rank's calls
@pytest.mark.parametrize("N,M", [(1, 1), (2, 2), (2, 4), (3, 2), (4, 3), (1, 16), (2, 6), (4, 8)])
@pytest.mark.parametrize("bits", [4, 8])
def test_local_calls_equal_the_ranks_row(N, M, bits):
    """The calls a real rank makes on its own buffers: step 1 on its bucket (whole and chunk
    by chunk), the fused hop on the chunks it receives, the final hop on the slices it
    receives -- each against the oracle, which gives the rank's row of the exchange."""
    from tests.test_oracle_pins import _received
    W = N * M
    for block, per_slice in ((64, 2 * 64), (512, 3 * 8192 + 512)):
        if W * W * per_slice > (1 << 23):
            per_slice = 2 * block
        E = W * per_slice
        g = inputs.draw("laplace", W * E, seed=3 * W + bits + block, dtype=torch.bfloat16,
                        device=DEV).reshape(W, E)
        c0, s0, c1, s1, out = oracle.qgz_pipeline(bits16(g), oracle.BF16, block, bits, N, M)
        for r in sorted({0, W - 1, W // 2}):
            lc, ls = zpp.qgz_reorder_quant_local(g[r], block, bits, N, M)
            assert np.array_equal(host(lc), c0[r]) and np.array_equal(host(ls), s0[r])
            pc = torch.full_like(lc, 0x5A)
            ps = torch.full_like(ls, -1.0)
            for p in range(M):
                zpp.qgz_reorder_quant_local(g[r], block, bits, N, M, pc, ps, chunks=(p, p + 1))
            assert torch.equal(pc, lc) and torch.equal(ps.view(torch.int32), ls.view(torch.int32))
            h1c, h1s, h2c, h2s = (torch.from_numpy(a).to(DEV) for a in
                                  _received(c0, s0, c1, s1, N, M, E, block, bits, r))
            oc, os_ = zpp.dequant_reduce_requant_local(h1c, h1s, E // M, block, bits, M)
            assert np.array_equal(host(oc), c1[r])
            assert np.array_equal(host(os_).view(np.uint32), s1[r].view(np.uint32))
            f = zpp.dequant_reduce_local(h2c, h2s, E // W, block, bits, N)
            assert_f32_parity(host(f), out[r])
            fa = zpp.dequant_reduce_local(h2c, h2s, E // W, block, bits, N, post_scale=1.0 / W,
                                          dtype=torch.bfloat16)
            want = oracle.dequant_reduce_chunks(h2c.cpu().numpy(), h2s.cpu().numpy(), E // W,
                                                block, bits, 1.0 / W, oracle.BF16)
            assert np.array_equal(bits16(fa), want)
    assert zb.zpp_device_fault() == 0


def _one_rank_exchange(port, q):
    import os
    import traceback
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import torch.distributed as dist
        from quantized_zero_communication_gb300 import exchange
        torch.cuda.set_device(0)
        dist.init_process_group("nccl", rank=0, world_size=1)
        groups = exchange.Groups(1, 1)
        g = inputs.draw("laplace", 8192, seed=2, dtype=torch.bfloat16, device="cuda:0")
        res = [exchange.qgz_step(g, 256, 4, groups, pipelined=p).cpu().numpy() for p in (0, 1)]
        dist.destroy_process_group()
        want = oracle.qgz_pipeline(bits16(g)[None], oracle.BF16, 256, 4, 1, 1)[4][0]
        ok = all(np.array_equal(r.view(np.uint32), want.view(np.uint32)) for r in res)
        q.put("ok" if ok else "owner slice differs from the oracle")
    except Exception:
        q.put(traceback.format_exc())


def test_exchange_step_on_one_nccl_rank():
    """The real-rank qgZ step (local kernels + NCCL collectives) on a world of one: both the
    all-to-all and the point-to-point hop-1 forms give the oracle's owner slice."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_one_rank_exchange, args=(port, q))
    p.start()
    msg = q.get(timeout=300)
    p.join(60)
    assert msg == "ok", msg
