"""Seeded synthetic inputs for the fused MoE expert GEMM + EP-combine path.

This package is shared by the CUDA path's harness and by the oracle. It draws
routing, gates and operand values and nothing else: it holds none of the
method's arithmetic (no row plan, no GEMM, no scatter, no signalling, no
combine).
"""

from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    Routing,
    make_routing,
    make_rank_values,
    make_layer_values,
    rows_per_rank,
    bf16_bits_from_f32,
    e4m3_bits_from_f32,
)
