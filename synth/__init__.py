"""Seeded synthetic inputs for the SeKV decode path and its cache build.

This package holds only input generation: random draws, the length mix of
surprisal-threshold spans, planted surprisal consistent with chosen spans,
low-rank-plus-noise key/value blocks, threshold placement with a margin, and
the packing of synthetic caches into the C-ABI layout.  It holds none of the
method's arithmetic (no segmentation, summaries, SVD, routing or attention):
both the CUDA path and the oracle consume what it produces.
"""

from .configs import CONFIGS, WorkloadConfig, get_config  # noqa: F401
from .gen import (  # noqa: F401
    span_lengths,
    planted_surprisal,
    lowrank_tokens,
    rank_budget_gates,
    query,
    routing_weights,
    build_inputs,
    decode_cache,
    pick_threshold,
    per_head_fraction,
    record_size,
    abi_to_numpy,
)
