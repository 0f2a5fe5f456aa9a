"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and
the benchmark.  This package holds no arithmetic of the aggregation or the
quantiser: it only draws graphs, features, weights and upstream gradients."""

from .graphs import (  # noqa: F401
    CONFIGS,
    Workload,
    make_workload,
    planted_partition_edges,
    dcsbm_edges,
    rmat_edges,
    circulant_edges,
    erdos_renyi_edges,
    star_edges,
    make_features,
    make_weight_bf16,
    bf16_bits_to_f32,
)
