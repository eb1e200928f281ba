"""Seeded synthetic inputs for low-bit MLA decode.

This package only draws random numbers and encodes them as bf16 bit patterns.
It holds none of the quantisation or attention arithmetic, so the CPU oracle
and the CUDA path can both be fed from it without sharing any of the method.
"""

from .synthetic import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    get,
    layout_of,
    make_paging,
    queries,
    sequence_lengths,
    sequence_tokens,
)
