"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers only: it holds none of the quantisation arithmetic.
Values are drawn in fp32 with a seeded ``torch.Generator`` on the requested device,
spiked where the workload asks for outliers, then cast to fp16/bf16 with
round-to-nearest-even (``Tensor.to``).

Workloads (the pages train GPT-style models on The Pile; no dataset is used here --
synthetic tensors with the shapes and value distributions below stand in for the
weights and gradients of those runs):

* qwZ round trip: fp16[1,048,576] ~ N(0, 0.02), 0.1 % of entries x20, seed 0.
* qgZ tiny topology: 2 nodes x 4 GPUs, bf16[8][65,536] ~ N(0, 1e-3), seed 1.
* qwZ on a GPT layer (hidden 8192): fp16 QKV 8192x24576, out-proj 8192x8192,
  MLP 8192x32768 and 32768x8192 (805,306,368 weights), ~ N(0, 0.02/sqrt(96)), seed 2.
* qgZ gradient bucket: bf16, 536,870,912 elements over 4 nodes x 8 GPUs
  (16,777,216 per rank), ~ Laplace(0, 1e-4), 0.01 % spikes x100, seed 3.
* sweep: sizes 2^20..2^30 (x4), fp16/bf16, bits {8,4}, block {64,256,1024,4096},
  N(0,0.02) / Laplace(0,1e-4) / U(-1,1) with 0.1 % x20 outliers, seed 100 + row.
"""
import math

import torch

GPT_LAYER_SHAPES = (("qkv", 8192, 24576), ("out_proj", 8192, 8192),
                    ("mlp_up", 8192, 32768), ("mlp_down", 32768, 8192))
GPT_LAYER_ELEMS = sum(a * b for _, a, b in GPT_LAYER_SHAPES)  # 805,306,368
GPT_SIGMA = 0.02 / math.sqrt(2 * 48)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(n, sigma, gen, device):
    return torch.randn(int(n), generator=gen, device=device, dtype=torch.float32) * sigma


def laplace(n, b, gen, device):
    """Inverse-CDF Laplace(0, b): u ~ U(-1/2, 1/2), x = -b sign(u) log1p(-2|u|).
    2|u| is capped just below 1 so the tail stays finite."""
    u = torch.rand(int(n), generator=gen, device=device, dtype=torch.float32) - 0.5
    t = torch.clamp(2.0 * u.abs(), max=1.0 - 2.0 ** -24)
    return -b * torch.sign(u) * torch.log1p(-t)


def uniform(n, lo, hi, gen, device):
    return torch.rand(int(n), generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo


def spike(x, frac, factor, gen):
    """Scale round(frac * n) seed-chosen entries (duplicates allowed) by `factor`."""
    n = x.numel()
    k = int(round(frac * n))
    if k:
        idx = torch.randint(0, n, (k,), generator=gen, device=x.device)
        x[idx] = x[idx] * factor
    return x


def draw(kind, n, seed, dtype, device="cpu"):
    """One of the sweep's distributions: 'normal' N(0,0.02), 'laplace' Laplace(0,1e-4),
    'uniform_outliers' U(-1,1) with 0.1 % of entries x20."""
    g = _gen(seed, device)
    if kind == "normal":
        x = normal(n, 0.02, g, device)
    elif kind == "laplace":
        x = laplace(n, 1e-4, g, device)
    elif kind == "uniform_outliers":
        x = spike(uniform(n, -1.0, 1.0, g, device), 1e-3, 20.0, g)
    else:
        raise ValueError(kind)
    return x.to(dtype)


def qwz_round_trip(device="cpu"):
    """fp16[1,048,576] ~ N(0, 0.02) with 0.1 % of entries x20 (seed 0)."""
    g = _gen(0, device)
    x = spike(normal(1 << 20, 0.02, g, device), 1e-3, 20.0, g)
    return x.to(torch.float16)


def qgz_tiny(device="cpu"):
    """2 nodes x 4 GPUs, bf16[8][65,536] ~ N(0, 1e-3) (seed 1)."""
    g = _gen(1, device)
    return normal(8 * 65536, 1e-3, g, device).to(torch.bfloat16).reshape(8, 65536)


def gpt_layer(device="cpu", div=1):
    """Flattened fp16 weights of one hidden-8192 GPT layer, ~ N(0, 0.02/sqrt(96))
    (seed 2). `div` shrinks every matrix's row count for profiling-sized runs."""
    g = _gen(2, device)
    n = GPT_LAYER_ELEMS // int(div)
    return normal(n, GPT_SIGMA, g, device).to(torch.float16)


def gradient_bucket(device="cpu", W=32, elems_per_rank=16_777_216):
    """bf16 [W][E] ~ Laplace(0, 1e-4) with 0.01 % spikes x100 (seed 3)."""
    g = _gen(3, device)
    x = spike(laplace(W * elems_per_rank, 1e-4, g, device), 1e-4, 100.0, g)
    return x.to(torch.bfloat16).reshape(W, elems_per_rank)


# The bucket's per-rank content as parameter gradients (for the fused flatten): 4083 rows
# of a 1024-wide embedding plus one transformer block of hidden 1024 (layer norms, QKV,
# attention output, a 4x MLP, with biases) -- 13 tensors, 16,777,216 elements per rank.
BUCKET_TENSOR_SHAPES = (
    ("embedding_rows", (4083, 1024)), ("ln1_weight", (1024,)), ("ln1_bias", (1024,)),
    ("qkv_weight", (3072, 1024)), ("qkv_bias", (3072,)), ("out_weight", (1024, 1024)),
    ("out_bias", (1024,)), ("ln2_weight", (1024,)), ("ln2_bias", (1024,)),
    ("fc1_weight", (4096, 1024)), ("fc1_bias", (4096,)), ("fc2_weight", (1024, 4096)),
    ("fc2_bias", (1024,)))


def bucket_tensor_sizes():
    """Elements per rank of each tensor of BUCKET_TENSOR_SHAPES, in order."""
    return [math.prod(shape) for _, shape in BUCKET_TENSOR_SHAPES]


def split_bucket(bucket, sizes):
    """[W][E] bucket -> one contiguous [W][n_t] tensor per size (consecutive column ranges:
    the tensors whose per-rank concatenation is the bucket)."""
    out, at = [], 0
    for n in sizes:
        out.append(bucket[:, at:at + n].contiguous())
        at += n
    assert at == bucket.shape[1]
    return out


def random_sizes(total, count, seed, unit=16):
    """`count` sizes, multiples of `unit` (0 allowed), summing to `total` (a multiple of
    `unit`): seeded uniform cut points."""
    g = _gen(seed, "cpu")
    cuts = torch.randint(0, total // unit + 1, (count - 1,), generator=g).sort().values * unit
    edges = [0] + cuts.tolist() + [total]
    return [b - a for a, b in zip(edges[:-1], edges[1:])]


SWEEP_SIZES = [1 << s for s in range(20, 31, 2)]
SWEEP_DTYPES = (torch.float16, torch.bfloat16)
SWEEP_BITS = (8, 4)
SWEEP_BLOCKS = (64, 256, 1024, 4096)
SWEEP_KINDS = ("normal", "laplace", "uniform_outliers")


def sweep_rows():
    """Rows of the sweep in enumeration order; row i uses seed 100 + i."""
    rows = []
    for size in SWEEP_SIZES:
        for dt in SWEEP_DTYPES:
            for bits in SWEEP_BITS:
                for block in SWEEP_BLOCKS:
                    for kind in SWEEP_KINDS:
                        rows.append(dict(size=size, dtype=dt, bits=bits, block=block,
                                         kind=kind, seed=100 + len(rows)))
    return rows
