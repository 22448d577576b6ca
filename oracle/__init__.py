"""CPU oracle for top-k sparse attention over a two-level KV cache.

TEST INFRASTRUCTURE: imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg.  It shares no code with the CUDA library.
"""
from .hisparse_oracle import (  # noqa: F401
    bf16_to_f64,
    indexer_scores,
    indexer_scores_many,
    indexer_scores_multihead,
    topk_select,
    page_bounds,
    page_scores,
    page_select,
    LRUHotCache,
    FIFOHotCache,
    RandomHotCache,
    splitmix64,
    belady_misses,
    sparse_attention,
    hot_over_full,
    hot_cache_bytes,
)
