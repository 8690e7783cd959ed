"""Pins for the CPU oracle: each test checks it against something other than itself --
hand-derived fixtures, IEEE conversions of independent libraries, closed-form error
bounds, exactly representable cases, brute-force placement on tiny topologies, and the
pages' qualitative claims (block-wise beats per-tensor; 4x less communication).

Pages: "ZeRO++: Extremely Efficient Collective Communication for Large Model Training"
(atlas.scime.ai summary: Approach, Measured effects table, Surprising findings);
"ZeRO++: Extremely Efficient Collective Communication for Giant Model Training"
(mlsanity.com, Abstract); "LIT-102: ZeRO++: ..." (Key takeaways).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_zero_communication_gb300 import inputs
from tests.golden import load_qgz_case, load_quant_cases

U = 2.0 ** -24  # unit roundoff of fp32


def bits16(t):
    """torch fp16/bf16 tensor -> numpy uint16 bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def f32_of_bits(b, dtype):
    t = torch.from_numpy(np.asarray(b, np.uint16).view(np.int16).copy())
    return t.view(torch.float16 if dtype == oracle.F16 else torch.bfloat16).float().numpy()


def unpack_codes(codes, n, bits):
    codes = np.asarray(codes, np.uint8)
    if bits == 8:
        return codes[:n].view(np.int8).astype(np.int64)
    lo = (codes & 0xF).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    q = np.empty(2 * codes.size, np.int64)
    q[0::2], q[1::2] = lo, hi
    q = q[:n]
    return np.where(q >= 8, q - 16, q)


# --------------------------------------------------------------------------- formats
def test_f16_to_f32_all_patterns_match_numpy():
    L = oracle.lib()
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([L.or_f16_to_f32(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_to_f32_all_patterns_match_torch():
    L = oracle.lib()
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([L.or_bf16_to_f32(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_probe_values():
    rng = np.random.default_rng(7)
    v = [rng.standard_normal(6000).astype(np.float32) * np.float32(s)
         for s in (1e-8, 1e-6, 1e-4, 1e-2, 1.0, 1e2, 1e4, 6e4)]
    # random bit patterns over the whole fp32 range (finite only)
    r = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    v.append(r[np.isfinite(r)])
    # exact ties between neighbouring fp16 / bf16 values, and the overflow edge
    h = np.arange(0, 0x7bff, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = np.arange(1, 0x7c00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    v.append(((h + h2) / 2).astype(np.float32))
    v.append(np.array([65504, 65519.996, 65520, 65536, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
                       2 ** -14, 2 ** -15 * 1.5, 0.0, -0.0], np.float32))
    b = (np.arange(0, 0x7f7f, 97, dtype=np.uint32) << 16).view(np.float32)
    v.append((b.view(np.uint32) | 0x8000).view(np.float32))  # bf16 ties
    v.append((b.view(np.uint32) | 0x18000).view(np.float32))
    v = np.concatenate(v)
    return np.concatenate([v, -v])


def test_f32_to_f16_rne_matches_numpy():
    L = oracle.lib()
    v = _f32_probe_values()
    ref = v.astype(np.float16).view(np.uint16)
    got = np.array([L.or_f32_to_f16(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_bf16_rne_matches_torch():
    L = oracle.lib()
    v = _f32_probe_values()
    ref = bits16(torch.from_numpy(v).to(torch.bfloat16))
    got = np.array([L.or_f32_to_bf16(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- fixtures
@pytest.mark.parametrize("case", load_quant_cases(), ids=lambda c: c["name"])
def test_golden_quant_cases(case):
    dt = oracle.F16 if case["dtype"] == "f16" else oracle.BF16
    tdt = torch.float16 if dt == oracle.F16 else torch.bfloat16
    x = torch.tensor(case["x"], dtype=torch.float64)
    xt = x.to(tdt)
    assert torch.equal(xt.double(), x), "fixture x must be exact in its dtype"
    codes, scales = oracle.quant_blockwise(bits16(xt), dt, case["block"], case["bits"])
    assert list(codes) == case["packed"]
    assert list(scales.view(np.uint32)) == case["scale_bits"]
    assert list(unpack_codes(codes, len(case["x"]), case["bits"])) == case["codes"]
    y = oracle.dequant_blockwise(codes, scales, len(case["x"]), case["block"], case["bits"], dt)
    want = bits16(torch.tensor(case["y"], dtype=torch.float64).to(tdt))
    assert np.array_equal(y, want)


# --------------------------------------------------------------------------- bounds
def _roundtrip_check(xbits, dt, block, bits):
    n = xbits.size
    qmax = 2 ** (bits - 1) - 1
    x = f32_of_bits(xbits, dt).astype(np.float64)
    codes, scales = oracle.quant_blockwise(xbits, dt, block, bits)
    assert codes.size == (n if bits == 8 else (n + 1) // 2)
    assert scales.size == -(-n // block)
    y = oracle.dequant_blockwise(codes, scales, n, block, bits, oracle.F32).astype(np.float64)
    s = np.repeat(scales.astype(np.float64), block)[:n]
    # the scale is the fp32 quotient of the block's absmax by qmax (within 1 ulp)
    pad = (-n) % block
    amax = np.abs(np.concatenate([x, np.zeros(pad)])).reshape(-1, block).max(1)
    nz = amax > 0
    assert np.all(np.abs(scales[nz] - amax[nz] / qmax) <= 2 * U * amax[nz] / qmax)
    assert np.all(scales[~nz] == 0)
    # per element: |x - q*s| <= s/2 + 3u|x| (scale, reciprocal and product roundings),
    # plus the fp32 rounding of y itself
    err = np.abs(x - y)
    bound = s / 2 + 4 * U * np.abs(x) + U * np.abs(y)
    assert np.all(err <= bound), float((err - bound).max())
    # the absmax element of every non-zero block lands on +-qmax
    q = unpack_codes(codes, n, bits)
    qpad = np.abs(np.concatenate([q, np.zeros(pad, np.int64)])).reshape(-1, block).max(1)
    assert np.all(qpad[nz] == qmax) and np.all(qpad[~nz] == 0)
    return x, y


@pytest.mark.parametrize("block", [64, 256, 1024, 4096])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("kind", inputs.SWEEP_KINDS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_round_trip_error_bound(block, bits, kind, dtype):
    n = 3 * 4096 + 1000 + 1  # several tiles, a ragged block and an odd tail
    t = inputs.draw(kind, n, seed=11, dtype=dtype)
    dt = oracle.F16 if dtype == torch.float16 else oracle.BF16
    _roundtrip_check(bits16(t), dt, block, bits)


def test_round_trip_qwz_config_and_fp16_output():
    t = inputs.qwz_round_trip()
    xb = bits16(t)
    x, _ = _roundtrip_check(xb, oracle.F16, 256, 8)
    codes, scales = oracle.quant_blockwise(xb, oracle.F16, 256, 8)
    y16 = oracle.dequant_blockwise(codes, scales, xb.size, 256, 8, oracle.F16)
    y = f32_of_bits(y16, oracle.F16).astype(np.float64)
    s = np.repeat(scales.astype(np.float64), 256)
    half_ulp16 = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64) / 2
    assert np.all(np.abs(x - y) <= s / 2 + 4 * U * np.abs(x) + half_ulp16 + U * np.abs(y))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_exactly_representable_blocks_round_trip_bit_exact(bits, dtype):
    """Values k*2^e with |k| <= qmax and one element at +-qmax*2^e: scale 2^e, inverse
    2^-e, codes k, so quant -> dequant returns the input bits unchanged."""
    qmax = 2 ** (bits - 1) - 1
    block, nblk = 64, 50
    rng = np.random.default_rng(3)
    k = rng.integers(-qmax, qmax + 1, (nblk, block))
    k[np.arange(nblk), rng.integers(0, block, nblk)] = qmax * rng.choice([-1, 1], nblk)
    e = rng.integers(-12, 4, nblk)[:, None]
    x = torch.from_numpy((k * np.exp2(e.astype(np.float64))).reshape(-1))
    xt = x.to(dtype)
    assert torch.equal(xt.double(), x)
    dt = oracle.F16 if dtype == torch.float16 else oracle.BF16
    codes, scales = oracle.quant_blockwise(bits16(xt), dt, block, bits)
    assert np.array_equal(scales.astype(np.float64), np.exp2(e[:, 0].astype(np.float64)))
    assert np.array_equal(unpack_codes(codes, x.numel(), bits), k.reshape(-1))
    y = oracle.dequant_blockwise(codes, scales, x.numel(), block, bits, dt)
    assert np.array_equal(y, bits16(xt))


def test_zero_block_gives_zero_scale_and_codes():
    x = np.zeros(300, np.uint16)
    x[256:] = bits16(torch.full((44,), 0.5, dtype=torch.float16))
    codes, scales = oracle.quant_blockwise(x, oracle.F16, 256, 4)
    assert scales[0] == 0 and np.all(codes[:128] == 0)
    assert scales[1] == np.float32(0.5) / np.float32(7)


def test_block_quant_is_local_so_shards_match_one_call():
    """qwZ quantises each rank's shard on its own; with block-aligned shards one call over
    the concatenation equals the per-shard calls (Approach: quantised all-gather)."""
    t = inputs.draw("normal", 16 * 2048 * 3, seed=5, dtype=torch.float16)
    xb = bits16(t)
    c_all, s_all = oracle.quant_blockwise(xb, oracle.F16, 2048, 8)
    parts = [oracle.quant_blockwise(p, oracle.F16, 2048, 8) for p in np.split(xb, 16)]
    assert np.array_equal(c_all, np.concatenate([p[0] for p in parts]))
    assert np.array_equal(s_all, np.concatenate([p[1] for p in parts]))


def test_blockwise_error_below_per_tensor_on_outlier_data():
    """Measured effects table / Surprising findings: non-blocked quantisation hurt
    convergence; LIT-102 Key takeaways: block-wise beats per-tensor. On the qwZ round-trip
    workload (0.1 % outliers x20) the blocked INT8 MSE must be below the per-tensor MSE."""
    xb = bits16(inputs.qwz_round_trip())
    n = xb.size
    x = f32_of_bits(xb, oracle.F16).astype(np.float64)
    res = {}
    for block in (256, n):
        c, s = oracle.quant_blockwise(xb, oracle.F16, block, 8)
        y = oracle.dequant_blockwise(c, s, n, block, 8, oracle.F32).astype(np.float64)
        res[block] = float(np.mean((x - y) ** 2))
    ratio = res[n] / res[256]
    print(f"per-tensor / block-256 MSE ratio = {ratio:.2f}")
    assert res[256] < res[n] and ratio > 2.0


def test_communication_volume_4x():
    """Abstract / summary: ZeRO-3 moves 3M per step (forward gather, backward gather,
    gradient reduce-scatter, fp16); ZeRO++ moves 0.5M (INT8 gather) + 0 (hpZ keeps the
    backward gather in the node) + 0.25M (INT4 gradients) = 0.75M cross-node: 4x less."""
    n = 1 << 20
    fp16_bytes = 2 * n
    c8, s8 = oracle.quant_blockwise(np.zeros(n, np.uint16), oracle.F16, 2048, 8)
    c4, s4 = oracle.quant_blockwise(np.zeros(n, np.uint16), oracle.F16, 2048, 4)
    assert c8.nbytes / fp16_bytes == 0.5 and c4.nbytes / fp16_bytes == 0.25
    assert s8.nbytes == 4 * (n // 2048)
    zero3 = 3 * fp16_bytes
    zpp = c8.nbytes + 0 + c4.nbytes
    assert zero3 / zpp == 4.0
    with_scales = c8.nbytes + s8.nbytes + c4.nbytes + s4.nbytes
    assert 3.98 < zero3 / with_scales < 4.0


# --------------------------------------------------------------------------- qgZ placement
TOPOS = [(1, 1), (1, 2), (2, 1), (2, 2), (2, 4), (3, 2), (4, 3)]


@pytest.mark.parametrize("N,M", TOPOS)
def test_reorder_places_every_reduced_slice_at_its_owner(N, M):
    """Approach (summary page): slices are reordered so that after the intra-node and the
    inter-node all-to-all every rank holds the reduction of its own slice. Brute force with
    small integers (exact fp32 sums), quantisation off."""
    W, S = N * M, 5
    E = W * S
    rng = np.random.default_rng(N * 10 + M)
    x = rng.integers(-50, 50, (W, E)).astype(np.float32)
    out = oracle.qgz_passthrough(x, N, M, reorder=True)
    want = np.stack([x[:, r * S:(r + 1) * S].sum(0) for r in range(W)])
    assert np.array_equal(out, want)
    if N > 1 and M > 1:
        bad = oracle.qgz_passthrough(x, N, M, reorder=False)
        assert not np.array_equal(bad, want)
        # without the reorder, rank (n, l) collects original slice l*N + n instead
        wrong = np.stack([x[:, (l * N + n) * S:(l * N + n + 1) * S].sum(0)
                          for n in range(N) for l in range(M)])
        assert np.array_equal(bad, wrong)


@pytest.mark.parametrize("N,M", TOPOS)
def test_reorder_is_a_slice_permutation(N, M):
    W, S = N * M, 3
    pos = [oracle.reorder_position(j, N, M) for j in range(W)]
    assert sorted(pos) == list(range(W))
    src = np.arange(W * S, dtype=np.float32)
    dst = oracle.reorder_slices(src, N, M)
    for j in range(W):
        assert np.array_equal(dst[pos[j] * S:(pos[j] + 1) * S], src[j * S:(j + 1) * S])
    # chunk l (N consecutive slices) holds exactly the slices owned by the ranks with
    # local index l, i.e. what local peer l reduces in the intra-node hop
    for l in range(M):
        owners = sorted(j for j in range(W) if pos[j] // N == l)
        assert owners == [n * M + l for n in range(N)]


@pytest.mark.parametrize("W", [1, 2, 6])
def test_flatten_bucket_inverts_the_split_into_tensors(W):
    """The fused flatten's definition: rank r's bucket is row r of every tensor, in tensor
    order. Cutting a bucket of distinct values (rank r, position i -> r * 10^6 + i) into
    consecutive column ranges and flattening again must give the bucket back; taking the
    tensors in another order, or the ranks' rows transposed, must not."""
    E = 400
    bucket = (np.arange(W)[:, None] * 10 ** 6 + np.arange(E)[None, :]).astype(np.float64)
    cuts = [0, 16, 16, 208, 400]  # one empty tensor
    tensors = [bucket[:, a:b].copy() for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.array_equal(oracle.flatten_bucket(tensors, W), bucket)
    assert not np.array_equal(oracle.flatten_bucket(tensors[::-1], W), bucket)
    if W > 1:
        flipped = [t.T.copy() for t in tensors]  # [n_t][W]: rank-minor, the wrong layout
        assert not np.array_equal(oracle.flatten_bucket(flipped, W), bucket)


def test_tensor_bucket_with_one_tensor_is_the_flat_call():
    x = inputs.draw("laplace", 4 * 2048, seed=5, dtype=torch.bfloat16).view(torch.int16).numpy()
    x = x.view(np.uint16).reshape(4, 2048)
    a = oracle.qgz_reorder_quant_tensors([x], oracle.BF16, 256, 4, 2, 2)
    b = oracle.qgz_reorder_quant(x, oracle.BF16, 256, 4, 2, 2)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


@pytest.mark.parametrize("N,M", [(1, 2), (2, 2), (2, 4), (1, 8), (4, 2)])
@pytest.mark.parametrize("bits", [4, 8])
def test_identical_exact_sources_reduce_exactly(N, M, bits):
    """Every rank holds the same exactly representable gradient (per-block k*2^e): each
    dequantised value is exact, fp32 sums of W equal terms are exact (W a power of two),
    and requantisation of M*k*2^e returns codes k with scale M*2^e. The final owner slice
    must be W times the rank's own slice, bit for bit."""
    W, B = N * M, 64
    qmax = 2 ** (bits - 1) - 1
    S = 2 * B
    E = W * S
    rng = np.random.default_rng(W + bits)
    nblk = E // B
    k = rng.integers(-qmax, qmax + 1, (nblk, B))
    k[np.arange(nblk), rng.integers(0, B, nblk)] = qmax
    e = rng.integers(-10, 0, nblk)[:, None]
    row = (k * np.exp2(e.astype(np.float64))).reshape(-1)
    g = torch.from_numpy(np.tile(row, (W, 1))).to(torch.bfloat16)
    assert torch.equal(g[0].double(), torch.from_numpy(row))
    c0, s0, c1, s1, out = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    want = (W * row).astype(np.float32).reshape(W, S)
    assert np.array_equal(out, want)
    # hop-1 scales are M times the source block scales of the same slices
    pos_s0 = s0[0].reshape(W, S // B)                 # scales by reordered slice position
    for n in range(N):
        for l in range(M):
            r = n * M + l
            chunk = pos_s0[l * N:(l + 1) * N].reshape(-1)
            assert np.array_equal(s1[r], (M * chunk.astype(np.float64)).astype(np.float32))


def _two_hop_bound(xs, N, M, block, bits):
    """Per-element bound on |final - direct sum| for every owner slice, computed from the
    original data only: two quantisations per value (source, after the intra-node sum)
    plus fp32 rounding. xs: fp64 [W][E]."""
    W, E = xs.shape
    S = E // W
    qmax = 2 ** (bits - 1) - 1
    nb = S // block
    bounds = np.empty((W, S))
    for r in range(W):
        sl = xs[:, r * S:(r + 1) * S]                                   # [W][S]
        amax1 = np.abs(sl).reshape(W, nb, block).max(2)
        s1 = np.repeat(amax1 / qmax * (1 + 2 * U), block, axis=1)       # [W][S]
        e1 = s1 / 2 + 4 * U * np.abs(sl)                                # source quantisation
        total = np.zeros(S)
        for n2 in range(N):
            rows = slice(n2 * M, (n2 + 1) * M)
            P = sl[rows].sum(0)                                         # intra-node sum
            E1 = e1[rows].sum(0) + M * U * np.abs(sl[rows]).sum(0) * 2  # + fp32 sum rounding
            amaxP = (np.abs(P) + E1).reshape(nb, block).max(1)
            s2 = np.repeat(amaxP / qmax * (1 + 2 * U), block)
            total += E1 + s2 / 2 + 4 * U * (np.abs(P) + E1)
        total += N * U * 2 * (np.abs(sl).sum(0) + total)                 # inter-node fp32 sum
        bounds[r] = total
    return bounds


@pytest.mark.parametrize("N,M,bits", [(2, 4, 4), (2, 4, 8), (4, 2, 4), (4, 2, 8)])
def test_two_hop_result_matches_direct_sum_within_two_quantisations(N, M, bits):
    """Approach: dequantise before reducing; LIT-102 Key takeaways: reduce locally in
    higher precision, a fixed number of quantisations per value. On the qgZ tiny workload
    (8 ranks, B=128; as 2 nodes x 4 GPUs and as 4 x 2, INT4 and INT8) every owner element
    is within the bound of the two quantisation steps of the direct sum over all ranks."""
    B = 128
    g = inputs.qgz_tiny()
    W, E = g.shape
    S = E // W
    xs = g.double().numpy()
    *_, out = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    direct = np.stack([xs[:, r * S:(r + 1) * S].sum(0) for r in range(W)])
    bound = _two_hop_bound(xs, N, M, B, bits)
    err = np.abs(out.astype(np.float64) - direct)
    assert np.all(err <= bound), float((err / bound).max())
    # the bound has teeth: a slice from the wrong owner, or a dropped source, breaks it
    assert np.any(np.abs(np.roll(out, 1, axis=0) - direct) > bound)
    dropped = np.stack([xs[1:, r * S:(r + 1) * S].sum(0) for r in range(W)])
    assert np.any(np.abs(dropped - direct) > bound)
    print(f"max err/bound = {float((err / bound).max()):.3f}")


def test_single_rank_requant_is_idempotent():
    """Topology 1x1: the intra-node hop requantises dequantised codes of one source; a
    block of q*s values has absmax qmax*s, so the codes come back unchanged."""
    g = inputs.draw("laplace", 4 * 1024, seed=9, dtype=torch.bfloat16).reshape(1, -1)
    c0, s0, c1, s1, out = oracle.qgz_pipeline(bits16(g), oracle.BF16, 256, 4, 1, 1)
    assert np.array_equal(c0, c1)
    rel = np.abs(s1.astype(np.float64) - s0) / np.maximum(s0, 1e-30)
    assert np.all(rel <= 2 * U)
    y = oracle.dequant_blockwise(c1[0], s1[0], g.shape[1], 256, 4, oracle.F32)
    assert np.array_equal(out[0], y)


def qgz_case_inputs(case):
    W, E = case["N"] * case["M"], case["elems_per_rank"]
    g = torch.zeros((W, E), dtype=torch.float64)
    for r, e, v in case["x"]:
        g[r, e] = v
    dt = torch.float16 if case["dtype"] == "f16" else torch.bfloat16
    gt = g.to(dt)
    assert torch.equal(gt.double(), g)
    return gt


def check_qgz_case(case, c0, s0, c1, s1, out):
    """Compare pipeline outputs with the sparse expectations of a fixture."""
    bits = case["bits"]
    for r, b, want in case["source_scale_bits"]:
        assert int(np.asarray(s0)[r, b:b + 1].view(np.uint32)[0]) == want
    for r, e, want in case["hop1_codes"]:
        assert unpack_codes(np.asarray(c1)[r], e + 1, bits)[e] == want
    for r, b, want in case["hop1_scale_bits"]:
        assert int(np.asarray(s1)[r, b:b + 1].view(np.uint32)[0]) == want
    o = np.asarray(out).copy()
    for r, e, want in case["out_bits"]:
        assert int(o[r, e:e + 1].view(np.uint32)[0]) == want, (r, e)
        o[r, e] = 0
    assert np.all(o == 0)


def test_golden_qgz_fused_sum():
    """Hand-derived 1x2 pipeline: each dequantised term enters the fp32 sum with one
    rounding (the fixture records the separately rounded alternative it excludes)."""
    case = load_qgz_case()
    g = qgz_case_inputs(case)
    dt = oracle.F16 if case["dtype"] == "f16" else oracle.BF16
    res = oracle.qgz_pipeline(bits16(g), dt, case["block"], case["bits"], case["N"], case["M"])
    check_qgz_case(case, *res)


def test_fixtures_exclude_the_separately_rounded_reading():
    """The two fused roundings of the oracle (the quantiser's exact product, one rounding
    per hop term) against the alternative that rounds every product to fp32 first. Both
    hand-derived fixtures are cases where the two readings differ: the alternative, redone
    here with numpy's IEEE fp32 operations, gives the excluded values the fixtures record
    (code 64, sum bits 0x3fa49249), and the oracle does not."""
    f32 = np.float32
    # int8_exact_product_tie: x = 1.5 in a block with amax 3.
    inv = f32(127) / f32(3)
    two_step = np.rint(f32(1.5) * inv)                     # the fp32 product is exactly 63.5
    assert f32(1.5) * inv == f32(63.5) and two_step == 64.0
    case = {c["name"]: c for c in load_quant_cases()}["int8_exact_product_tie"]
    xt = torch.tensor(case["x"], dtype=torch.float64).to(torch.float16)
    codes, _ = oracle.quant_blockwise(bits16(xt), oracle.F16, case["block"], case["bits"])
    got = unpack_codes(codes, len(case["x"]), 8)
    assert got[1] == 63 and got[1] != two_step and got[2] == -63
    # qgz_fused_sum: hop-1 element 0 is 2 s + 7 s with s = fl32(1/7).
    s = f32(1) / f32(7)
    separate = f32(f32(2) * s) + f32(f32(7) * s)           # two roundings of the second term
    assert separate.view(np.uint32) == 0x3fa49249
    fused = f32(float(s) * 9.0)                             # 2 s + 7 s is exact in double
    assert fused.view(np.uint32) == 0x3fa4924a
    qcase = load_qgz_case()
    g = qgz_case_inputs(qcase)
    dt = oracle.F16 if qcase["dtype"] == "f16" else oracle.BF16
    s1 = oracle.qgz_pipeline(bits16(g), dt, qcase["block"], qcase["bits"], qcase["N"],
                             qcase["M"])[3]
    # the hop-1 block scale is fl32(sum / 7): 0x3e3c14e7 from the fused sum, 0x3e3c14e6
    # from the separately rounded one
    got = np.asarray(s1)[0, 0:1].view(np.uint32)[0]
    assert (fused / f32(7)).view(np.uint32) == got == 0x3e3c14e7
    assert (separate / f32(7)).view(np.uint32) == 0x3e3c14e6


@pytest.mark.parametrize("N,M", [(2, 2), (2, 4), (1, 8)])
def test_average_of_identical_exact_sources_is_the_own_slice(N, M):
    """The abstract describes the gradient step as an average: with every rank holding the
    same exactly representable gradient, the averaged owner slice (post_scale 1/W, W a power
    of two) is the rank's own slice, exactly, in fp32 and after the bf16 cast."""
    W, B, bits = N * M, 64, 4
    qmax = 7
    S = 2 * B
    E = W * S
    rng = np.random.default_rng(100 + W)
    nblk = E // B
    k = rng.integers(-qmax, qmax + 1, (nblk, B))
    k[np.arange(nblk), rng.integers(0, B, nblk)] = -qmax
    e = rng.integers(-6, 2, nblk)[:, None]
    row = (k * np.exp2(e.astype(np.float64))).reshape(-1)
    g = torch.from_numpy(np.tile(row, (W, 1))).to(torch.bfloat16)
    c0, s0, c1, s1, _ = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    avg = oracle.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, 1.0 / W, oracle.F32)
    assert np.array_equal(avg, row.astype(np.float32).reshape(W, S))
    avg16 = oracle.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, 1.0 / W, oracle.BF16)
    assert np.array_equal(avg16, bits16(torch.from_numpy(row).to(torch.bfloat16)).reshape(W, S))


def test_averaged_two_hop_with_an_inexact_average_within_bound():
    """W = 6 (3 nodes x 2 GPUs): 1/W is not a power of two, so post_scale = fp32(1/6) carries
    one rounding (<= u relative) on top of the product's own (<= u): the averaged owner
    slices stay within the two-quantisation bound / W of the direct average plus 2u."""
    N, M, B, bits = 3, 2, 128, 4
    W = N * M
    E = W * B * 8
    g = inputs.draw("laplace", W * E, seed=61, dtype=torch.bfloat16).reshape(W, E)
    S = E // W
    xs = g.double().numpy()
    c0, s0, c1, s1, total = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    direct = np.stack([xs[:, r * S:(r + 1) * S].sum(0) for r in range(W)]) / W
    bound = _two_hop_bound(xs, N, M, B, bits) / W
    ps = float(np.float32(1.0 / W))
    avg = oracle.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, ps, oracle.F32).astype(np.float64)
    assert np.all(np.abs(avg - direct) <= bound + 2 * U * np.abs(avg) + 1e-30)
    # the average is the sum times fp32(1/W), rounded once: exactly fp32(total * ps)
    assert np.array_equal(avg.astype(np.float32), (total.astype(np.float64) * ps).astype(np.float32))


def test_averaged_two_hop_result_within_bound():
    """The averaged (1/W) owner slices of the 2 x 4 workload stay within the two-quantisation
    bound of the direct average, in fp32 and after a bf16 cast (plus half a bf16 ulp)."""
    N, M, B, bits = 2, 4, 128, 4
    g = inputs.qgz_tiny()
    W, E = g.shape
    S = E // W
    xs = g.double().numpy()
    c0, s0, c1, s1, total = oracle.qgz_pipeline(bits16(g), oracle.BF16, B, bits, N, M)
    direct = np.stack([xs[:, r * S:(r + 1) * S].sum(0) for r in range(W)]) / W
    bound = _two_hop_bound(xs, N, M, B, bits) / W
    avg = oracle.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, 1.0 / W, oracle.F32).astype(np.float64)
    assert np.all(np.abs(avg - direct) <= bound + U * np.abs(avg))
    a16 = f32_of_bits(oracle.dequant_reduce_scaled(c1, s1, E, B, bits, N, M, 1.0 / W, oracle.BF16),
                      oracle.BF16).astype(np.float64)
    half_ulp = np.abs(a16) * 2.0 ** -8
    assert np.all(np.abs(a16 - direct) <= bound + U * np.abs(avg) + half_ulp)


# --------------------------------------------------------------------------- received chunks
def _received(c0, s0, c1, s1, N, M, E, block, bits, r):
    """The buffers rank r receives in the two hops of the virtual layout: chunk l of its
    node's ranks (local-index order), then slice n of the hop-1 outputs of ranks (n', l)."""
    W, C, S = N * M, E // M, E // (N * M)
    n, l = divmod(r, M)
    cbC, cbS = oracle.code_bytes(C, bits), oracle.code_bytes(S, bits)
    h1c = np.stack([c0[n * M + j][l * cbC:(l + 1) * cbC] for j in range(M)])
    h1s = np.stack([s0[n * M + j][l * (C // block):(l + 1) * (C // block)] for j in range(M)])
    h2c = np.stack([c1[j * M + l][n * cbS:(n + 1) * cbS] for j in range(N)])
    h2s = np.stack([s1[j * M + l][n * (S // block):(n + 1) * (S // block)] for j in range(N)])
    return h1c, h1s, h2c, h2s


@pytest.mark.parametrize("N,M", [(1, 2), (2, 2), (2, 4), (3, 2), (1, 3), (4, 1)])
@pytest.mark.parametrize("bits", [4, 8])
def test_one_receivers_hops_equal_its_row_of_the_exchange(N, M, bits):
    """The per-receiver hop functions, fed the chunks / slices the exchange delivers, give
    the receiver's row of the whole-exchange functions (which are pinned above by
    placement, error bounds and the fixture): the index maps of the two formulations agree."""
    W, block = N * M, 64
    E = W * 3 * block
    g = inputs.draw("laplace", W * E, seed=70 + W + bits, dtype=torch.bfloat16).reshape(W, E)
    c0, s0, c1, s1, out = oracle.qgz_pipeline(bits16(g), oracle.BF16, block, bits, N, M)
    avg = oracle.dequant_reduce_scaled(c1, s1, E, block, bits, N, M, 1.0 / W, oracle.BF16)
    for r in range(W):
        h1c, h1s, h2c, h2s = _received(c0, s0, c1, s1, N, M, E, block, bits, r)
        oc, os_ = oracle.dequant_reduce_requant_chunks(h1c, h1s, E // M, block, bits)
        assert np.array_equal(oc, c1[r]) and np.array_equal(os_.view(np.uint32),
                                                            s1[r].view(np.uint32))
        f = oracle.dequant_reduce_chunks(h2c, h2s, E // W, block, bits)
        assert np.array_equal(f.view(np.uint32), out[r].view(np.uint32))
        fa = oracle.dequant_reduce_chunks(h2c, h2s, E // W, block, bits, 1.0 / W, oracle.BF16)
        assert np.array_equal(fa, avg[r])


@pytest.mark.parametrize("bits", [4, 8])
def test_one_chunk_reduces_to_its_dequantisation(bits):
    """With one source the hop-2 sum is fma(q, s, +0) = fl32(q * s), the dequantisation."""
    x = inputs.draw("uniform_outliers", 4 * 256, seed=5, dtype=torch.float16)
    codes, scales = oracle.quant_blockwise(bits16(x), oracle.F16, 256, bits)
    got = oracle.dequant_reduce_chunks(codes[None], scales[None], x.numel(), 256, bits)
    want = oracle.dequant_blockwise(codes, scales, x.numel(), 256, bits, oracle.F32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("K", [2, 4, 8])
def test_identical_exact_chunks_sum_exactly(K):
    """K identical chunks whose terms are exact small multiples of a power-of-two scale:
    every sum is K times the term exactly, and the requantised block keeps the codes with
    K times the scale."""
    block, bits = 64, 4
    q = np.tile(np.array([7, -7, 3, 0, -1, 5, 2, -4], np.int64), 2 * block // 8)
    nib = (q & 0xF).astype(np.uint8)
    codes = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    scales = np.full(2, 2.0 ** -10, np.float32)
    ch = np.stack([codes] * K), np.stack([scales] * K)
    total = oracle.dequant_reduce_chunks(*ch, 2 * block, block, bits)
    assert np.array_equal(total, (K * q * 2.0 ** -10).astype(np.float32))
    oc, os_ = oracle.dequant_reduce_requant_chunks(*ch, 2 * block, block, bits)
    assert np.array_equal(oc, codes) and np.all(os_ == np.float32(K * 2.0 ** -10))
