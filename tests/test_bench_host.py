"""Host-side logic of bench.py: the byte accounting, the multi-rank timing helpers (two
gloo ranks on the CPU), and the reference arm's JSON line."""
import json
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def test_step_bytes_match_the_workload_arithmetic():
    n, E = bench.workload_sizes(1)
    b = bench.step_bytes(n, E)
    # qwZ INT8 block 2048: 2 B read + 1 B codes + 4/2048 B scale per element
    assert b["K1_quant"] == 2 * n + n + 4 * n // 2048
    assert abs(b["K1_quant"] / n - 3.00195) < 1e-5
    # fused hop: reads 512 Mi INT4 codes + scales (272.6 MB), writes 1/8 of that (34.1 MB)
    assert abs(b["K4_dequant_reduce_requant"] / 1e6 - 306.7) < 0.1
    W = 32
    assert b["K3_reorder_quant"] == W * E * 2 + W * E // 2 + 4 * W * E // 512
    assert b["K5_dequant_reduce"] == W * (E // 8 // 2 + 4 * (E // 8) // 512) + 4 * E
    assert sum(b.values()) == sum(bench.step_bytes(*bench.workload_sizes(1)).values())


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w = bench.init_dist("gloo")
    bench.barrier()
    m = bench.max_over_ranks(10.0 * (rank + 1))
    bench.barrier()
    q.put((r, w, m))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert res == [(0, 2, 20.0), (1, 2, 20.0)]


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_prints_the_contract_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-seconds", "0.5"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["qgz_topology"] == [4, 8]


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_rejects_short_warmup():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
