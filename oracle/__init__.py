"""fp64 CPU oracle for blockwise Ring Self-Attention.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU
baseline of the benchmark are the only callers.  The CUDA library never
imports, links or runs anything from this package, and this package imports
nothing from the library.
"""
from .oracle import (  # noqa: F401
    build,
    fwd,
    fwd_rows,
    bwd,
    bwd_rows,
    ring_fwd,
    ring_step,
    ring_step_bwd,
    merge,
    ffn,
    ffn_bwd,
    owner_rank,
    ring_sources,
    dfa_schedule,
    SCHEDULES,
    visible_pairs,
)
