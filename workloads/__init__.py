"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests/bench.

This package only draws random numbers and rounds them to bf16 storage; it holds none of
the FP8 recipes' arithmetic, so both sides of a parity test can take their inputs from it.
"""
from .generators import (  # noqa: F401
    bf16_bits_normal,
    bf16_bits_from_f32,
    bf16_bits_to_f32,
    sigma_schedule,
    workload_shapes,
    STREAM_X, STREAM_W, STREAM_DY, STREAM_W2, STREAM_OUTLIER, STREAM_SIGMA, STREAM_STEP0,
)
