"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package only draws random data in the shapes and distributions of the
routed-MoE prefill workloads.  It holds none of the method's arithmetic: no
dequantisation, routing, sorting, GEMM, activation or combine.
"""

from .inputs import *  # noqa: F401,F403
