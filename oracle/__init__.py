"""CPU oracle for the IndexCache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code with the CUDA library or its Python binding; it reads the raw input
bytes (bf16 / e4m3 bit patterns, fp32 values) copied to host memory and
computes every step in float64 with NumPy.
"""

from .indexcache import (  # noqa: F401
    bf16_to_f64,
    e4m3_to_f64,
    dequantize_e4m3,
    indexer_scores,
    topk_positions,
    indexer_topk,
    schedule,
    schedule_rows,
    sparse_attention,
    forward_pattern,
    PatternError,
    validate_pattern,
    overlap,
    greedy_full_layers,
)
