"""Positional LSH oracle (test infrastructure only).

A plain, slow, fp64 CPU statement of the approximate-ALiBi hot path, written
from "Positional LSH: Binary Block Matrix Approximation for Attention with
Linear Biases" (Wolfson & Wagner), technical summary, Methodology items 1-3.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library.
"""
from .oracle import (  # noqa: F401
    build,
    philox4x32_10,
    ln64,
    draw,
    bins_one,
    sample_bins,
    bins_fixed,
    share_groups,
    bias_error,
    plsh_attn_rows,
    plsh_attn_backward,
    plsh_parts_rows,
    alibi_exact_rows,
    set_threads,
    max_threads,
    all_rows,
)
