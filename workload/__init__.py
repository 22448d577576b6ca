"""Seeded synthetic inputs for one decode step of top-k sparse attention over a
two-level (host DRAM + HBM hot cache) KV store.

This package generates inputs only: it holds no scoring, selection, cache or
attention arithmetic, so the CPU oracle and the CUDA library can both be fed
from it without sharing any of the method's code.
"""
from .synth import (  # noqa: F401
    Workload,
    WORKLOADS,
    make_workload,
    stress_point,
    f32_to_bf16_bits,
    prefill_kv,
    prefill_idx_keys,
    query_walk,
    query_walk_heads,
    step_idx_weights,
    step_query,
    step_kv_row,
    step_idx_key,
    kv_rows_at,
    idx_keys_upto,
    STRESS_B,
    STRESS_SIGMA,
)
