"""Seeded synthetic inputs for the sparse paged decode-attention path.

This package is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark.  It only draws random numbers and lays them out (paged K/V storage,
page tables, queries); it computes nothing that the method itself computes
(no summaries, bounds, selection, softmax or quantisation).
"""

from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    DRIFT_SIGMA,
    make_inputs,
    make_layout,
    make_layer,
    drift_queries,
    generator,
)
