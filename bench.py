"""Benchmark of the ZeRO++ block-quantisation hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  qwZ on one hidden-8192 GPT layer (805,306,368 fp16 weights, 16 virtual ranks, INT8
  block 2048): K1 quantise, K2 dequantise the gathered codes;
  qgZ on one gradient bucket (536,870,912 bf16 gradients over 4 nodes x 8 GPUs, INT4
  block 512): K3 reorder + quantise, K4 fused dequant -> fp32 sum -> requant (K = 8),
  K5 final dequant-reduce (K = 4).
Metric: algorithmic bytes moved per second (GB/s) -- reads plus writes each kernel
must make, summed over the step -- with the dominant kernel's fraction of the measured
HBM bandwidth. Inputs (5.4 GB) far exceed the 129 MB L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica on its own GPU (weak scaling, no
data-path collective); rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quant / dequant-reduce-requant GB/s and % of GB300 HBM peak (1 GPU)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

# Workload (sizes of the qwZ GPT-layer and qgZ bucket configurations).
QWZ_BLOCK, QWZ_BITS = 2048, 8
QGZ_N, QGZ_M, QGZ_BLOCK, QGZ_BITS = 4, 8, 512, 4
QGZ_ELEMS_PER_RANK = 16_777_216
KERNELS = ("K1_quant", "K2_dequant", "K3_reorder_quant", "K4_dequant_reduce_requant",
           "K5_dequant_reduce")
KERNEL_SOURCES = {"K1_quant": ["quant.cu", "quant_tile.cuh", "zpp_device.cuh"],
                  "K2_dequant": ["dequant.cu", "zpp_device.cuh"],
                  "K3_reorder_quant": ["reorder_quant.cu", "quant_tile.cuh", "zpp_device.cuh"],
                  "K4_dequant_reduce_requant": ["qgz.cu", "zpp_device.cuh"],
                  "K5_dequant_reduce": ["qgz.cu", "zpp_device.cuh"]}
# The kernels held to the throughput target (80 % of the measured HBM bandwidth at 256M
# elements and more): quantise (K1, and K3 for the gradients), dequantise (K2) and the fused
# dequant-reduce-requant (K4).
TARGET_KERNELS = ("K1_quant", "K2_dequant", "K3_reorder_quant", "K4_dequant_reduce_requant")


# ----------------------------------------------------------------------------- accounting
def code_bytes(n, bits):
    return n if bits == 8 else (n + 1) // 2


def step_bytes(n_qwz, E, div=1):
    """Algorithmic bytes per launch of each kernel (reads + writes it cannot avoid)."""
    W, M = QGZ_N * QGZ_M, QGZ_M
    C, S = E // M, E // W
    qs = 4 * math.ceil(n_qwz / QWZ_BLOCK)
    b = {
        "K1_quant": 2 * n_qwz + code_bytes(n_qwz, QWZ_BITS) + qs,
        "K2_dequant": code_bytes(n_qwz, QWZ_BITS) + qs + 2 * n_qwz,
        "K3_reorder_quant": W * (2 * E + code_bytes(E, QGZ_BITS) + 4 * (E // QGZ_BLOCK)),
        "K4_dequant_reduce_requant": W * (code_bytes(E, QGZ_BITS) + 4 * (E // QGZ_BLOCK))
        + W * (code_bytes(C, QGZ_BITS) + 4 * (C // QGZ_BLOCK)),
        "K5_dequant_reduce": W * (code_bytes(C, QGZ_BITS) + 4 * (C // QGZ_BLOCK)) + 4 * W * S,
    }
    return b


def step_elements(n_qwz, E):
    """Input elements per launch of each kernel (for elements/s)."""
    W, M = QGZ_N * QGZ_M, QGZ_M
    return {"K1_quant": n_qwz, "K2_dequant": n_qwz, "K3_reorder_quant": W * E,
            "K4_dequant_reduce_requant": W * E, "K5_dequant_reduce": W * (E // M)}


def workload_sizes(div):
    from quantized_zero_communication_gb300 import inputs
    return inputs.GPT_LAYER_ELEMS // div, QGZ_ELEMS_PER_RANK // div


def workload_config(div, n_qwz, E):
    return {
        "workload": "qwZ GPT layer (hidden 8192: 805,306,368 fp16 weights, 16 virtual ranks, "
                    "INT8 block 2048) + qgZ gradient bucket (536,870,912 bf16 over 4 nodes x "
                    "8 GPUs, INT4 block 512, K=8 then K=4)" + (f", sizes / {div}" if div > 1 else ""),
        "qwz_elements": n_qwz, "qwz_block": QWZ_BLOCK, "qwz_bits": QWZ_BITS, "qwz_ranks": 16,
        "qgz_elements": QGZ_N * QGZ_M * E, "qgz_topology": [QGZ_N, QGZ_M],
        "qgz_block": QGZ_BLOCK, "qgz_bits": QGZ_BITS,
        "l2": "inputs larger than L2 (no flush)", "parallelism": "replica per GPU",
    }


# ----------------------------------------------------------------------------- distributed
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), \
        int(os.environ.get("WORLD_SIZE", 1))


def init_dist(backend):
    import torch.distributed as dist
    rank, _, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value, device="cpu"):
    """Largest `value` over all ranks (the value itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    FLAGS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id, self.proc, self.file = gpu_id, None, None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_id)], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        rows = []
        with open(self.file.name) as f:
            for line in f:
                p = [c.strip() for c in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(p[1]), float(p[2]), p[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside:  # region shorter than the sampling period: nearest samples
            mid = (t0 + t1) / 2
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
        sm = sorted(r[1] for r in inside)
        reasons = sorted({name for r in inside for name, v in zip(self.FLAGS, r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "source": "nvidia-smi"}


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (the driver's libnvidia-ml, read
    only) about every millisecond in a thread, so a timed region of a few tens of ms still
    gets tens of samples. start() returns False when NVML is not usable here."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid):
        self.uuid, self.rows, self.thread, self.stop_flag = uuid, [], None, False

    def start(self):
        import ctypes
        import threading
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if L.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
                return False
            get_reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # 1 = SM clock
                return False
        except (OSError, AttributeError):
            return False
        self.max_mhz = float(mx.value)

        def run():
            mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self.stop_flag:
                if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                        get_reasons(h, ctypes.byref(rs)) == 0:
                    self.rows.append((time.time(), float(mhz.value), int(rs.value)))
                time.sleep(0.001)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()
        return True

    def stop(self, t0, t1):
        self.stop_flag = True
        self.thread.join(2)
        if not self.rows:
            return None
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        if not inside:  # region shorter than the sampling period: the nearest samples
            mid = (t0 + t1) / 2
            inside = sorted(self.rows, key=lambda r: abs(r[0] - mid))[:2]
        sm = sorted(r[1] for r in inside)
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items()
                          if r[2] & bit})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(inside), "source": "nvml"}


# ----------------------------------------------------------------------------- peaks
# GB300 HBM3e nominal bandwidth (the spec figure), reported beside the measured denominator
SPEC_HBM_GBS = 7900.0


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "quantized_zero_communication_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, units_ratio):
    """Per-launch DRAM bytes of `kernel` from the committed ncu capture, scaled to this
    launch's size; None if no capture exists or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_digest") != source_digest(kernel):
        return None
    return rec["dram_bytes_per_launch"] * units_ratio / rec.get("units_ratio", 1.0)


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import quantized_zero_communication_gb300 as zpp
    from quantized_zero_communication_gb300 import build as zbuild, inputs

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    if not os.path.exists(zbuild.LIB):
        zbuild.build()
    div = args.size_div
    n_qwz, E = workload_sizes(div)
    W, N, M = QGZ_N * QGZ_M, QGZ_N, QGZ_M
    C, S = E // M, E // W
    per_kernel_bytes = step_bytes(n_qwz, E)
    bytes_step = sum(per_kernel_bytes.values())

    # Inputs resident in HBM; outputs preallocated.
    x = inputs.gpt_layer(dev, div=div)
    g = inputs.gradient_bucket(dev, W=W, elems_per_rank=E)
    codes = torch.empty(code_bytes(n_qwz, QWZ_BITS), dtype=torch.uint8, device=dev)
    scales = torch.empty(math.ceil(n_qwz / QWZ_BLOCK), dtype=torch.float32, device=dev)
    y = torch.empty(n_qwz, dtype=torch.float16, device=dev)
    c0 = torch.empty((W, code_bytes(E, QGZ_BITS)), dtype=torch.uint8, device=dev)
    s0 = torch.empty((W, E // QGZ_BLOCK), dtype=torch.float32, device=dev)
    c1 = torch.empty((W, code_bytes(C, QGZ_BITS)), dtype=torch.uint8, device=dev)
    s1 = torch.empty((W, C // QGZ_BLOCK), dtype=torch.float32, device=dev)
    out = torch.empty((W, S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    B = {"x": x, "g": g, "codes": codes, "scales": scales, "y": y, "c0": c0, "s0": s0,
         "c1": c1, "s1": s1, "out": out}
    calls = {
        "K1_quant": lambda: zpp.quant_blockwise(B["x"], QWZ_BLOCK, QWZ_BITS, B["codes"], B["scales"]),
        "K2_dequant": lambda: zpp.dequant_blockwise(B["codes"], B["scales"], n_qwz, QWZ_BLOCK,
                                                    QWZ_BITS, y=B["y"]),
        "K3_reorder_quant": lambda: zpp.qgz_reorder_quant(B["g"], QGZ_BLOCK, QGZ_BITS, N, M,
                                                          B["c0"], B["s0"]),
        "K4_dequant_reduce_requant": lambda: zpp.dequant_reduce_requant(
            B["c0"], B["s0"], E, QGZ_BLOCK, QGZ_BITS, N, M, B["c1"], B["s1"]),
        "K5_dequant_reduce": lambda: zpp.dequant_reduce(B["c1"], B["s1"], E, QGZ_BLOCK, QGZ_BITS,
                                                        N, M, B["out"]),
    }
    uses = {"K1_quant": ("x", "codes", "scales"), "K2_dequant": ("codes", "scales", "y"),
            "K3_reorder_quant": ("g", "c0", "s0"), "K4_dequant_reduce_requant": ("c0", "s0", "c1", "s1"),
            "K5_dequant_reduce": ("c1", "s1", "out")}
    active = KERNELS
    if args.only:
        for k in KERNELS:  # one pass fills every intermediate, then keep the kernel's own
            calls[k]()
        torch.cuda.synchronize()
        active = tuple(k for k in KERNELS if k.startswith(args.only))
        del x, g, codes, scales, y, c0, s0, c1, s1, out
        for name in list(B):
            if name not in uses[active[0]]:
                del B[name]
        torch.cuda.empty_cache()
        bytes_step = sum(per_kernel_bytes[k] for k in active)

    def step(ev=None):
        for i, k in enumerate(active):
            if ev is not None:
                ev[i].record(stream)
            calls[k]()
        if ev is not None:
            ev[len(active)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # Timed region: exactly K steps, events on the launching stream around each kernel.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(active) + 1)]
              for _ in range(args.steps)]
    sampler = NvmlClockSampler(_smi_id(dev, local))
    if not sampler.start():
        sampler = ClockSampler(_smi_id(dev, local))
        sampler.start()
    time.sleep(0.15)
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for k in range(args.steps):
        step(events[k])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    elapsed_ms = start.elapsed_time(end)
    max_ms = max_over_ranks(elapsed_ms, device=dev)
    ms_per_step = max_ms / args.steps
    value = world * bytes_step * args.steps / (max_ms * 1e-3) / 1e9

    # Per-kernel durations (ms, summed over the timed steps).
    kt = {k: 0.0 for k in active}
    for ev in events:
        for i, k in enumerate(active):
            kt[k] += ev[i].elapsed_time(ev[i + 1])
    peak, peak_src = hbm_peak()
    kernels = {}
    for k in active:
        avg_s = kt[k] / args.steps * 1e-3
        gbs = per_kernel_bytes[k] / avg_s / 1e9
        kernels[k] = {"us": round(avg_s * 1e6, 2), "bytes": per_kernel_bytes[k],
                      "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                      "gelem_per_s": round(step_elements(n_qwz, E)[k] / avg_s / 1e9, 1),
                      "share": round(kt[k] / sum(kt.values()), 4)}
    dom = max(active, key=lambda k: kt[k])
    full_bytes = step_bytes(*workload_sizes(1))[dom]
    roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak,
            "peak_source": peak_src, "unit": "GB/s",
            "frac": round(kernels[dom]["gbs"] / peak, 4),
            "traffic": ncu_traffic(dom, per_kernel_bytes[dom] / full_bytes),
            "spec_peak": SPEC_HBM_GBS, "frac_spec": round(kernels[dom]["gbs"] / SPEC_HBM_GBS, 4)}
    # same-run copy kernel on 1 GiB (reference for the same HBM)
    copy_gbs = None if args.only else _copy_reference(zpp, torch, dev)
    if copy_gbs:
        for k in active:
            kernels[k]["frac_same_run_copy"] = round(kernels[k]["gbs"] / copy_gbs, 4)
        roof["frac_same_run_copy"] = kernels[dom]["frac_same_run_copy"]
    # The copy peak is a 1:1 read/write stream; a kernel whose mix is 2:1 or 1:2 can move
    # more bytes per second than it, so a fraction above 1 is possible and is flagged here.
    roof["peak_exceeded"] = kernels[dom]["gbs"] > peak
    targets = [k for k in TARGET_KERNELS if k in active]
    weakest = min(targets, key=lambda k: kernels[k]["gbs"] / peak) if targets else None
    roof_min = None if weakest is None else {
        "kernel": weakest, "achieved": kernels[weakest]["gbs"], "peak": peak, "unit": "GB/s",
        "frac": kernels[weakest]["frac"], "spec_peak": SPEC_HBM_GBS,
        "frac_spec": round(kernels[weakest]["gbs"] / SPEC_HBM_GBS, 4),
        "frac_same_run_copy": kernels[weakest].get("frac_same_run_copy")}
    overlap = None if args.only else _qgz_overlap(zpp, torch, dev, g, E, c0, s0, c1, s1, out,
                                                  per_kernel_bytes)
    as_tensors = None if args.only else _qgz_tensors(zpp, torch, dev, g, E, c0, s0,
                                                     per_kernel_bytes)

    result = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
              "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
              "data": "synthetic (seeded N(0,0.02/sqrt(96)) fp16 weights; Laplace(0,1e-4) bf16 "
                      "gradients with 0.01% x100 spikes)",
              "config": workload_config(div, n_qwz, E),
              "roofline": roof, "roofline_min": roof_min, "kernels": kernels,
              "copy_kernel_gbs": round(copy_gbs, 1) if copy_gbs else None,
              "qgz_pipelined": overlap, "qgz_tensors": as_tensors,
              "gpu_launches": len(active) * args.steps, "clocks": clocks}
    # The metric's two named parts: quantise (qwZ K1) and dequant-reduce-requant (K4).
    for key, k in (("quant", "K1_quant"), ("drr", "K4_dequant_reduce_requant")):
        if k in kernels:
            result[f"{key}_gbs"] = kernels[k]["gbs"]
            result[f"{key}_frac"] = kernels[k]["frac"]
            result[f"{key}_gelem_per_s"] = kernels[k]["gelem_per_s"]
    if args.only:
        result["only"] = active[0]
    if not args.no_e2e and not args.only:
        result["e2e"] = run_e2e(args, zpp, torch, dev, x, g, codes, scales, y, c0, s0, c1, s1,
                                out, n_qwz, E, bytes_step, world, pieces=args.e2e_pieces)
    B.clear()
    if not args.only:
        del x, g, codes, scales, y, c0, s0, c1, s1, out
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


def _smi_id(dev, local):
    import torch
    u = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if u is not None:
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(local)


def _copy_reference(zpp, torch, dev):
    a = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    for _ in range(3):
        zpp.device_copy(a, b)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(10):
        zpp.device_copy(a, b)
    e.record()
    torch.cuda.synchronize()
    t = s.elapsed_time(e) / 10 * 1e-3
    del a, b
    return 2 * (1 << 30) / t / 1e9


def _qgz_overlap(zpp, torch, dev, g, E, c0, s0, c1, s1, out, per_kernel_bytes, reps=20):
    """The qgZ half (K3 -> K4 -> K5) timed as three whole-exchange launches and as M
    independent local-index sub-pipelines spread over side streams, where one chunk's
    ALU-bound fused hop overlaps another chunk's memory-bound reorder+quantise."""
    N, M = QGZ_N, QGZ_M
    stream = torch.cuda.current_stream(dev)
    bufs = zpp.QgzBuffers(c0, s0, c1, s1, out)
    qbytes = sum(per_kernel_bytes[k] for k in KERNELS[2:])

    def serial():
        zpp.qgz_reorder_quant(g, QGZ_BLOCK, QGZ_BITS, N, M, c0, s0)
        zpp.dequant_reduce_requant(c0, s0, E, QGZ_BLOCK, QGZ_BITS, N, M, c1, s1)
        zpp.dequant_reduce(c1, s1, E, QGZ_BLOCK, QGZ_BITS, N, M, out)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    res = {"serial_us": round(timed(serial), 1)}
    for n_streams in (2, 4):
        streams = [torch.cuda.Stream(dev) for _ in range(n_streams)]
        us = timed(lambda: zpp.qgz_pipelined(g, QGZ_BLOCK, QGZ_BITS, N, M, bufs=bufs,
                                             streams=streams))
        res[f"pipelined_{n_streams}_streams_us"] = round(us, 1)
    lo, hi = torch.cuda.Stream(dev, priority=0), torch.cuda.Stream(dev, priority=-1)
    for chunks in (1, 2):
        us = timed(lambda: zpp.qgz_pipelined(g, QGZ_BLOCK, QGZ_BITS, N, M, bufs=bufs,
                                             streams=("split", lo, hi), chunks=chunks))
        res[f"pipelined_split_priority_{chunks}_chunk_us"] = round(us, 1)
    best = min(v for k, v in res.items() if k.startswith("pipelined"))
    res["gbs_serial"] = round(qbytes / (res["serial_us"] * 1e-6) / 1e9, 1)
    res["gbs_pipelined"] = round(qbytes / (best * 1e-6) / 1e9, 1)
    return res


def _qgz_tensors(zpp, torch, dev, g, E, c0, s0, per_kernel_bytes, reps=20):
    """K3 on the bucket given as its parameter-gradient tensors (13 per rank): the fused
    flatten against flattening first (torch.cat into the [W][E] bucket) and then K3."""
    from quantized_zero_communication_gb300 import inputs
    N, M = QGZ_N, QGZ_M
    sizes = inputs.bucket_tensor_sizes()
    if sum(sizes) != E:  # a reduced workload (--size-div): same tensor count, scaled
        sizes = [s * E // sum(sizes) // 16 * 16 for s in sizes[:-1]]
        sizes.append(E - sum(sizes))
    tensors = inputs.split_bucket(g, sizes)
    stream = torch.cuda.current_stream(dev)

    def fused():
        zpp.qgz_reorder_quant_tensors(tensors, QGZ_BLOCK, QGZ_BITS, N, M, c0, s0)

    def flatten_then_k3():
        torch.cat(tensors, dim=1, out=g)
        zpp.qgz_reorder_quant(g, QGZ_BLOCK, QGZ_BITS, N, M, c0, s0)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    us_fused, us_flat = timed(fused), timed(flatten_then_k3)
    del tensors
    return {"tensors": len(sizes), "fused_us": round(us_fused, 1),
            "flatten_then_k3_us": round(us_flat, 1),
            "fused_gbs": round(per_kernel_bytes["K3_reorder_quant"] / (us_fused * 1e-6) / 1e9, 1)}


def run_e2e(args, zpp, torch, dev, x, g, codes, scales, y, c0, s0, c1, s1, out, n_qwz, E,
            bytes_step, world, pieces=2):
    """The same step through the public API with host buffers: every step copies the
    weights and gradients in from pinned host memory and copies the dequantised weights
    and the reduced gradient slices back out. All host-to-device copies run in order on one
    input stream -- the weights in `pieces` block-aligned pieces (each its own pinned
    allocation), then the gradients; each weight piece is quantised, dequantised and copied
    back on a second stream as soon as it has arrived, and the gradient half runs on a
    third, so copies back overlap the copies in of later data."""
    N, M = QGZ_N, QGZ_M
    per = n_qwz // pieces
    assert per % QWZ_BLOCK == 0 and per * pieces == n_qwz
    nb = per // QWZ_BLOCK

    def pinned(shape, dtype):
        return torch.empty(shape, dtype=dtype, pin_memory=True)

    # The device-only results of the timed region, to check the end-to-end outputs against.
    y_ref, out_ref = y.clone(), out.clone()
    hx = [pinned((per,), x.dtype) for _ in range(pieces)]
    hy = [pinned((per,), y.dtype) for _ in range(pieces)]
    for i in range(pieces):
        hx[i].copy_(x[i * per:(i + 1) * per])
    hg, hout = pinned(g.shape, g.dtype), pinned(out.shape, out.dtype)
    hg.copy_(g)
    main = torch.cuda.current_stream(dev)
    s_in, s_w, s_g = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def step():
        fork = torch.cuda.Event()
        fork.record(main)
        for st in (s_in, s_w, s_g):
            st.wait_event(fork)
        arrived = []
        with torch.cuda.stream(s_in):
            for i in range(pieces):
                x[i * per:(i + 1) * per].copy_(hx[i], non_blocking=True)
                arrived.append(torch.cuda.Event())
                arrived[-1].record(s_in)
            g.copy_(hg, non_blocking=True)
            g_in = torch.cuda.Event()
            g_in.record(s_in)
        with torch.cuda.stream(s_w):  # qwZ: each weight piece as soon as it is on the device
            for i in range(pieces):
                lo, hi = i * per, (i + 1) * per
                s_w.wait_event(arrived[i])
                zpp.quant_blockwise(x[lo:hi], QWZ_BLOCK, QWZ_BITS, codes[lo:hi],
                                    scales[i * nb:(i + 1) * nb])
                zpp.dequant_blockwise(codes[lo:hi], scales[i * nb:(i + 1) * nb], per, QWZ_BLOCK,
                                      QWZ_BITS, y=y[lo:hi])
                hy[i].copy_(y[lo:hi], non_blocking=True)
        with torch.cuda.stream(s_g):  # qgZ: once the gradients are on the device
            s_g.wait_event(g_in)
            zpp.qgz_reorder_quant(g, QGZ_BLOCK, QGZ_BITS, N, M, c0, s0)
            zpp.dequant_reduce_requant(c0, s0, E, QGZ_BLOCK, QGZ_BITS, N, M, c1, s1)
            zpp.dequant_reduce(c1, s1, E, QGZ_BLOCK, QGZ_BITS, N, M, out)
            hout.copy_(out, non_blocking=True)
        for st in (s_in, s_w, s_g):
            join = torch.cuda.Event()
            join.record(st)
            main.wait_event(join)

    steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(main)
    for _ in range(steps):
        step()
    e.record(main)
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (*hx, hg))
    d2h = sum(t.numel() * t.element_size() for t in (*hy, hout))
    # What came back through the host buffers must be what the device-only path computed.
    same = all(torch.equal(hy[i].to(dev), y_ref[i * per:(i + 1) * per]) for i in range(pieces))
    same = same and torch.equal(hout.to(dev), out_ref)
    if not same:
        raise RuntimeError("end-to-end outputs differ from the device-only path")
    return {"value": round(world * bytes_step * steps / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 3), "streams": 3, "weight_pieces": pieces,
            "checked": True}


# ----------------------------------------------------------------------------- oracle legs
def oracle_sample_step(div, seed_cache={}):
    """The whole path on the CPU oracle over a 1/div sample of the workload (the first
    1/div of the layer's weights; the bucket with 1/div of the elements per rank on the
    same 4 x 8 topology). Returns (algorithmic bytes, seconds)."""
    import numpy as np
    import torch
    import oracle
    from quantized_zero_communication_gb300 import inputs

    key = div
    if key not in seed_cache:
        seed_cache.clear()
        x = inputs.gpt_layer("cpu", div=div)
        g = inputs.gradient_bucket("cpu", W=QGZ_N * QGZ_M, elems_per_rank=QGZ_ELEMS_PER_RANK // div)
        seed_cache[key] = (x.view(torch.int16).numpy().view(np.uint16),
                           g.view(torch.int16).numpy().view(np.uint16))
    xb, gb = seed_cache[key]
    n_qwz, E = xb.size, gb.shape[1]
    t0 = time.perf_counter()
    c, s = oracle.quant_blockwise(xb, oracle.F16, QWZ_BLOCK, QWZ_BITS)
    oracle.dequant_blockwise(c, s, n_qwz, QWZ_BLOCK, QWZ_BITS, oracle.F16)
    oracle.qgz_pipeline(gb, oracle.BF16, QGZ_BLOCK, QGZ_BITS, QGZ_N, QGZ_M)
    dt = time.perf_counter() - t0
    return sum(step_bytes(n_qwz, E).values()), dt


def _calibrated_div(target_s):
    """Smallest power-of-two divisor (>= 1) whose sample runs in about target_s seconds,
    and the time one such sample is predicted to take."""
    div = 1024
    b, t = oracle_sample_step(div)
    while div > 1 and t * 2 < target_s:
        div //= 2
        t *= 2
    return div, t


def cpu_baseline(target_s):
    """The oracle, as it stands, on all host cores over a bounded sample of the workload:
    a 1/div slice, repeated when even the whole workload takes less than target_s."""
    import oracle
    cores = oracle.set_threads(len(os.sched_getaffinity(0)))
    div, t_pred = _calibrated_div(target_s)
    reps = max(1, int(target_s / max(t_pred, 1e-3))) if div == 1 else 1
    tot_b, tot_t = 0, 0.0
    for _ in range(reps):
        b, t = oracle_sample_step(div)
        tot_b += b
        tot_t += t
    what = "the whole workload" if div == 1 else (
        f"1/{div} of the workload (first 1/{div} of the layer weights; bucket with "
        f"{QGZ_ELEMS_PER_RANK // div} elements per rank, same topology)")
    # the same oracle on one core, over a smaller sample (about a fifth of the time)
    oracle.set_threads(1)
    div1, _ = _calibrated_div(max(target_s / 5, 0.5))
    b1, t1 = oracle_sample_step(div1)
    oracle.set_threads(cores)
    return {"value": round(tot_b / tot_t / 1e9, 3), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": f"{what}, {reps} pass(es), {tot_t:.1f} s",
            "single_core": {"value": round(b1 / t1 / 1e9, 3), "unit": UNIT,
                            "sample": f"1/{div1} of the workload, {t1:.1f} s"}}


def run_reference(args):
    """The oracle timed as the reference arm (rank 0 only)."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    import oracle
    cores = oracle.set_threads(len(os.sched_getaffinity(0)))
    per_step = args.ref_seconds or max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    div, _ = _calibrated_div(per_step)
    for _ in range(args.warmup):
        oracle_sample_step(div)
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_sample_step(div)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    n_qwz, E = workload_sizes(1)
    sample = (f"each step 1/{div} of the workload (first 1/{div} of the layer weights; bucket "
              f"with {QGZ_ELEMS_PER_RANK // div} elements per rank, same 4x8 topology)")
    result = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
              "ms_per_step": round(tot_t / args.steps * 1e3, 2), "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "f32",
              "data": "synthetic (same generators and seeds as the GPU arm)",
              "config": workload_config(1, n_qwz, E),
              "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                               "kind": "oracle", "sample": sample},
              "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                      "d2h_bytes_per_step": 0}}
    print(json.dumps(result), flush=True)
    return result


def run_sweep(args):
    """Times K1, K2 and the fused K-way hop (topology 1 x K, K in {2, 8, 16}) over the
    sweep's sizes x dtypes x bits x blocks (N(0, 0.02) data; timing does not depend on the
    values): 20 launches after 3 warm-up ones, back to back between one pair of events when
    the buffers exceed the 129 MB L2, else one by one with a 256 MiB write flushing L2
    before each."""
    import torch
    import quantized_zero_communication_gb300 as zpp
    from quantized_zero_communication_gb300 import build as zbuild, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if not os.path.exists(zbuild.LIB):
        zbuild.build()
    peak, peak_src = hbm_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, small):
        for _ in range(3):
            fn()
        if not small:  # buffers larger than L2: 20 launches back to back, one event pair
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / 20 * 1e-3
        tot = 0.0
        for _ in range(20):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        return tot / 20 * 1e-3

    def pick(values, chosen):
        return [v for v in values if not chosen or v in chosen]

    dtypes = [d for d in inputs.SWEEP_DTYPES
              if not args.sweep_dtypes or str(d).replace("torch.", "") in args.sweep_dtypes]
    rows = []
    for size in pick(inputs.SWEEP_SIZES, [1 << e for e in args.sweep_log2 or []]):
        for dt in dtypes:
            x = inputs.draw("normal", size, seed=100, dtype=dt, device=dev)
            for bits in pick(inputs.SWEEP_BITS, args.sweep_bits):
                for block in pick(inputs.SWEEP_BLOCKS, args.sweep_blocks):
                    cb, ns = code_bytes(size, bits), math.ceil(size / block)
                    codes, scales = zpp.quant_blockwise(x, block, bits)
                    y = torch.empty_like(x)
                    small = 2 * size < L2_BYTES * 2
                    t1 = timed(lambda: zpp.quant_blockwise(x, block, bits, codes, scales), small)
                    t2 = timed(lambda: zpp.dequant_blockwise(codes, scales, size, block, bits, y=y),
                               small)
                    b12 = 2 * size + cb + 4 * ns
                    row = {"size": size, "dtype": str(dt).replace("torch.", ""), "bits": bits,
                           "block": block,
                           "quant_us": round(t1 * 1e6, 1), "quant_frac": round(b12 / t1 / 1e9 / peak, 3),
                           "dequant_us": round(t2 * 1e6, 1), "dequant_frac": round(b12 / t2 / 1e9 / peak, 3)}
                    if dt == torch.bfloat16:
                        for K in pick((2, 8, 16), args.sweep_k):
                            E = size // K
                            if E % (K * block):
                                continue
                            c0, s0 = zpp.qgz_reorder_quant(x.view(K, E), block, bits, 1, K)
                            c1, s1 = zpp.dequant_reduce_requant(c0, s0, E, block, bits, 1, K)
                            t4 = timed(lambda: zpp.dequant_reduce_requant(c0, s0, E, block, bits, 1,
                                                                          K, c1, s1), small)
                            b4 = (cb + 4 * ns) * (1 + 1 / K)
                            row[f"drr_K{K}_us"] = round(t4 * 1e6, 1)
                            row[f"drr_K{K}_frac"] = round(b4 / t4 / 1e9 / peak, 3)
                            del c0, s0, c1, s1
                    rows.append(row)
                    del codes, scales, y
            del x
            torch.cuda.empty_cache()
    print(json.dumps({"sweep": rows, "peak": peak, "peak_source": peak_src}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--size-div", type=int, default=1,
                    help="shrink the workload by this power of two (profiling runs only)")
    ap.add_argument("--sweep", action="store_true",
                    help="time quant, dequant and the fused hop over the sweep's sizes, dtypes, "
                         "widths and blocks (one JSON object; not the benchmark line)")
    ap.add_argument("--sweep-log2", type=int, nargs="*",
                    help="with --sweep: only these sizes (log2 of the element count)")
    ap.add_argument("--sweep-bits", type=int, nargs="*", help="with --sweep: only these widths")
    ap.add_argument("--sweep-blocks", type=int, nargs="*", help="with --sweep: only these blocks")
    ap.add_argument("--sweep-dtypes", nargs="*", help="with --sweep: float16 and/or bfloat16")
    ap.add_argument("--sweep-k", type=int, nargs="*", help="with --sweep: fused-hop K values")
    ap.add_argument("--only", choices=("K1", "K2", "K3", "K4", "K5"),
                    help="time one kernel of the step on the full workload, keeping only its "
                         "own buffers on the device (profiling runs)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-pieces", type=int, default=2,
                    help="weight pieces of the end-to-end leg (1, 2, 4 or 8)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=0.0,
                    help="target seconds per reference step (default: fit the run in minutes)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.size_div < 1 or args.size_div & (args.size_div - 1) or args.size_div > 1024:
        ap.error("--size-div must be a power of two <= 1024")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
