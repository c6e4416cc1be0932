"""Seeded synthetic inputs for decode-step KV-cache attention.

This package is the only code shared by the CUDA path's harness (tests, bench)
and the CPU oracle.  It draws numbers and lays out workload structure (shapes,
current positions, block tables, residency masks, prefix-sharing groups); it
holds none of the method's arithmetic: no slot mapping, no attended set, no
RoPE, no softmax.

Values are N(0, 1) draws from torch's generator, seeded per
(workload seed, layer, stream, token owner, block of 256 positions), so any
position of any sequence can be drawn on its own and the same position always
gets the same value, whichever range it was requested in.
"""

from .generator import POSITION_BLOCK, derive_seed, randn, to_dtype
from .workloads import (
    Workload,
    WORKLOAD_NAMES,
    make_workload,
    tiny_ring_sink_f32,
    ring_bf16,
    sink_window_bf16,
    paged_shared_prefix_bf16,
    long_context_pool_bf16,
    ring_int8,
    sink_window_int8,
    paged_shared_prefix_int8,
    as_int8,
)

__all__ = [
    "POSITION_BLOCK",
    "derive_seed",
    "randn",
    "to_dtype",
    "Workload",
    "WORKLOAD_NAMES",
    "make_workload",
    "tiny_ring_sink_f32",
    "ring_bf16",
    "sink_window_bf16",
    "paged_shared_prefix_bf16",
    "long_context_pool_bf16",
    "ring_int8",
    "sink_window_int8",
    "paged_shared_prefix_int8",
    "as_int8",
]
