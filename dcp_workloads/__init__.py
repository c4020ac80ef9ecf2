"""Seeded synthetic workloads for DCP decode attention.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds no arithmetic of the method itself: it only draws random numbers,
rounds them to the storage dtype with library casts, lays tokens out densely
per request, hands out physical block ids from a random permutation once a
caller has said how many blocks each (rank, request) needs, draws the
candidate positions a sparse-attention indexer would select, and builds one
deterministic peaked input (a strongly attended key above a long flat tail).
"""

from .configs import CONFIGS, CONFIG_ORDER, config
from .gen import Workload, allocate_blocks, bf16_bits, fp8_bits, make_workload, sink_tail_workload, sparse_candidates

__all__ = [
    "CONFIGS",
    "CONFIG_ORDER",
    "config",
    "Workload",
    "make_workload",
    "allocate_blocks",
    "bf16_bits",
    "fp8_bits",
    "sink_tail_workload",
    "sparse_candidates",
]
