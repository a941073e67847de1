"""Seeded synthetic workloads for routing attention.

This package only draws inputs: random token vectors, values and initial
centroids with the shapes and value structure of the routing-attention
workloads, plus the bf16 storage format.  It holds none of the method's
arithmetic (no routing, scoring, selection, attention or centroid update), so
that the CUDA library and the fp64 oracle can both be fed from it without
sharing any of the computation they are compared on.
"""

from .synth import (  # noqa: F401
    CONFIGS,
    CONFIG_ORDER,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_workload,
    make_random,
    workload_name,
)
