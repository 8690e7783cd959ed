"""GB300 (sm_103a) ZeRO++ block-quantisation hot path: qwZ quantise / dequantise and
the qgZ reorder-quantise, fused intra-node dequant-reduce-requant and final
dequant-reduce, behind the C ABI declared in ``include/zpp.h``.

``binding`` is the ctypes layer over ``libzpp.so``; ``inputs`` holds the seeded
synthetic workloads. The library is loaded on first use.
"""
from .binding import (  # noqa: F401
    Topology, ZppError, dequant_blockwise, dequant_reduce, dequant_reduce_local,
    dequant_reduce_requant, dequant_reduce_requant_local, dequant_reduce_scaled, device_copy,
    LocalRange, QgzBuffers, qgz_pipelined, qgz_reorder_quant, qgz_reorder_quant_local,
    qgz_reorder_quant_tensors, quant_blockwise, zpp_code_bytes, zpp_num_scales,
    zpp_status_string)
