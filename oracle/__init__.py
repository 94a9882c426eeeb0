"""CPU oracle for the FP8 linear-layer hot path.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the benchmark's
CPU-baseline leg. The CUDA path never imports it and it never imports the CUDA path.
"""
from . import fp8_oracle  # noqa: F401
