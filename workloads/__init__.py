"""Seeded synthetic workloads for wave-index decode attention.

This package holds only input generation (random draws, shapes, bf16 casts of
the drawn inputs).  It contains none of the method's arithmetic: the index
build and the tripartite attention live in the CUDA library and, separately,
in the CPU oracle.  Both sides receive the arrays produced here.
"""

from .synthetic import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits,
    bf16_bits_to_float32,
    generate,
    retrieval_budget,
)
