"""The data plane across real ranks (exchange.py), run as 2 and 4 gloo ranks on the CPU.

Every rank builds the same seeded workload, computes its own step with the CPU oracle and
moves the bytes with the exchange layer. Each buffer a rank receives must equal, bit for
bit, the slices of the single-process virtual layout that the kernels read there (chunk l
of the node's ranks in hop 1, slice n of the local index's hop-1 outputs in hop 2, the
whole quantised weight set after the qwZ gather), and the oracle's per-receiver hops on
those buffers must give the rank's row of the single-process result. Both hop-1 forms are
checked: one all-to-all, and point-to-point transfers in ring order with the chunks
produced one at a time."""
import os
import socket
import traceback

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from quantized_zero_communication_gb300 import exchange, inputs

B = 64


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _rank_checks(rank, N, M, bits):
    W = N * M
    n, l = divmod(rank, M)
    S = 2 * B                      # slice: two blocks
    E, C = W * S, N * S
    cbC, cbS = oracle.code_bytes(C, bits), oracle.code_bytes(S, bits)
    groups = exchange.Groups(N, M)

    # the virtual layout, as the single-process run sees it
    g = inputs.draw("laplace", W * E, seed=40 + W + bits, dtype=torch.bfloat16).reshape(W, E)
    c0, s0, c1, s1, out = oracle.qgz_pipeline(_bits16(g), oracle.BF16, B, bits, N, M)

    # step 1 of this rank (its row; the reorder does not depend on the rank)
    codes, scales = torch.from_numpy(c0[rank].copy()), torch.from_numpy(s0[rank].copy())

    # hop 1: chunk l of ranks (n, 0..M-1), local-index order
    want_c = np.stack([c0[n * M + j][l * cbC:(l + 1) * cbC] for j in range(M)])
    want_s = np.stack([s0[n * M + j][l * (C // B):(l + 1) * (C // B)] for j in range(M)])
    rc, rs = exchange.hop1_all_to_all(codes, scales, groups)
    assert np.array_equal(rc.numpy(), want_c), "hop-1 all-to-all codes"
    assert np.array_equal(rs.numpy().view(np.uint32), want_s.view(np.uint32)), "hop-1 scales"

    # the same by point-to-point, each chunk produced just before it is sent
    pc, ps = torch.zeros_like(codes), torch.zeros_like(scales)
    order = []

    def produce(p):
        order.append(p)
        pc[p * cbC:(p + 1) * cbC] = codes[p * cbC:(p + 1) * cbC]
        ps[p * (C // B):(p + 1) * (C // B)] = scales[p * (C // B):(p + 1) * (C // B)]

    qc, qs = exchange.hop1_p2p(pc, ps, groups, produce_chunk=produce)
    assert order == [(l + d) % M for d in range(M)]
    assert torch.equal(qc, rc) and torch.equal(qs.view(torch.int32), rs.view(torch.int32))

    # the fused hop on what arrived == this rank's row of the virtual hop 1
    oc, os_ = oracle.dequant_reduce_requant_chunks(rc.numpy(), rs.numpy(), C, B, bits)
    assert np.array_equal(oc, c1[rank]), "hop-1 codes"
    assert np.array_equal(os_.view(np.uint32), s1[rank].view(np.uint32)), "hop-1 scales"

    # hop 2: slice n of the hop-1 outputs of ranks (0..N-1, l)
    want2_c = np.stack([c1[j * M + l][n * cbS:(n + 1) * cbS] for j in range(N)])
    want2_s = np.stack([s1[j * M + l][n * (S // B):(n + 1) * (S // B)] for j in range(N)])
    r2c, r2s = exchange.hop2_all_to_all(torch.from_numpy(oc), torch.from_numpy(os_), groups)
    assert np.array_equal(r2c.numpy(), want2_c), "hop-2 codes"
    assert np.array_equal(r2s.numpy().view(np.uint32), want2_s.view(np.uint32)), "hop-2 scales"
    final = oracle.dequant_reduce_chunks(r2c.numpy(), r2s.numpy(), S, B, bits)
    assert np.array_equal(final.view(np.uint32), out[rank].view(np.uint32)), "owner slice"

    # qwZ: quantise the shard, gather codes + scales == the whole weight set quantised
    shard = 3 * 256
    x = inputs.draw("normal", W * shard, seed=60 + W, dtype=torch.float16)
    xb = _bits16(x)
    sc, ss = oracle.quant_blockwise(xb[rank * shard:(rank + 1) * shard], oracle.F16, 256, 8)
    gc, gs = exchange.qwz_all_gather(torch.from_numpy(sc), torch.from_numpy(ss))
    fc, fs = oracle.quant_blockwise(xb, oracle.F16, 256, 8)
    assert np.array_equal(gc.numpy(), fc), "qwZ gathered codes"
    assert np.array_equal(gs.numpy().view(np.uint32), fs.view(np.uint32)), "qwZ gathered scales"
    full = oracle.dequant_blockwise(gc.numpy(), gs.numpy(), W * shard, 256, 8, oracle.F16)

    # hpZ: keep slice l of the full weights; the intra-node gather gives them back
    full_t = torch.from_numpy(full.view(np.int16).copy()).view(torch.float16)
    sec = exchange.hpz_secondary(full_t, groups)
    assert sec.numel() == W * shard // M
    back = exchange.hpz_all_gather(sec, groups)
    assert torch.equal(back.view(torch.int16), full_t.view(torch.int16)), "hpZ gather"


def _rank_main(rank, world, port, N, M, bits, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
        _rank_checks(rank, N, M, bits)
        torch.distributed.barrier()
        q.put((rank, "ok"))
    except Exception:  # report to the parent instead of hanging the other ranks
        q.put((rank, traceback.format_exc()))
    finally:
        if torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


def _run(N, M, bits):
    world = N * M
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, N, M, bits, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(60)
        if p.is_alive():
            p.kill()
    bad = {r: v for r, v in res.items() if v != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{v}" for r, v in bad.items())


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,M", [(1, 2), (2, 1)])
def test_exchange_two_ranks(N, M, bits):
    _run(N, M, bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,M", [(2, 2), (1, 4), (4, 1)])
def test_exchange_four_ranks(N, M, bits):
    _run(N, M, bits)
