"""Seeded synthetic inputs for paged decode.

This package is shared by the CUDA path's tests and benchmark and by the CPU
oracle.  It draws random numbers and sizes buffers; it holds none of the
method's arithmetic (no block allocation, no slot computation, no attention).
"""

from .synth import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits,
    context_lens,
    free_order,
    normal,
    pool_blocks,
    queries,
    random_pool,
    serving_step_tokens,
)
