"""Seeded synthetic inputs shared by the CPU oracle, the tests and the benchmark.

This package draws random numbers and shapes them into the workloads the
serving path is exercised on (queries, keys, values, page tables, sequence
lengths). It holds none of the quantisation method's arithmetic: no rotation,
clipping, quantisation, packing or attention lives here, so neither side of a
parity test can inherit a mistake from it.
"""

from .generators import (  # noqa: F401
    WorkloadSpec,
    WORKLOADS,
    bf16_round,
    bf16_bits,
    kv_outlier_channels,
    query_basis,
    draw_kv,
    draw_queries,
    draw_shared_direction_qk,
    draw_page_pool,
    draw_ragged_lengths,
)
