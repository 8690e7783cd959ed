"""The GPU arm of bench.py keeps its JSON contract: one line with every key the driver
reads, on a reduced workload (sizes / 64) so that it runs in seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--size-div", "64", "--steps", "5",
                        "--warmup", "3", "--e2e-steps", "3", "--cpu-seconds", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert "workload" in d["config"]
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["achieved"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert "traffic" in roof
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["checked"] is True  # host outputs equal the device-only path's, bit for bit
    # the weakest of the target kernels, and the metric's two named parts
    assert roof["spec_peak"] == 7900.0 and abs(roof["frac_spec"] - roof["achieved"] / 7900.0) < 1e-3
    rmin = d["roofline_min"]
    targets = ("K1_quant", "K2_dequant", "K3_reorder_quant", "K4_dequant_reduce_requant")
    assert rmin["kernel"] in targets
    assert rmin["frac"] == min(d["kernels"][k]["frac"] for k in targets)
    assert d["quant_gbs"] == d["kernels"]["K1_quant"]["gbs"]
    assert d["drr_gbs"] == d["kernels"]["K4_dequant_reduce_requant"]["gbs"]
    assert isinstance(roof["peak_exceeded"], bool)
    assert d["gpu_launches"] == 5 * d["steps"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert set(d["kernels"]) == {"K1_quant", "K2_dequant", "K3_reorder_quant",
                                 "K4_dequant_reduce_requant", "K5_dequant_reduce"}
