"""CPU oracle of the quantized MoE expert-FFN layer (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use
this package.  It is a plain single-threaded binary64 implementation in C
(moe_oracle.c) that shares no code with the CUDA library; this module only
marshals numpy arrays into it.
"""
from .oracle import *  # noqa: F401,F403
