"""Seeded synthetic inputs for the lazy loop step (shapes and random draws only)."""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    active_count,
    key_count,
    prefill_loops,
    decode_context,
    decode_token_loops,
    normal_bf16,
    BLOCK_FF_MULT,
    block_weights,
    block_input,
)
