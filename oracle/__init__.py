"""CPU oracle for the weight-only NVFP4 (W4A16) MoE layer -- TEST INFRASTRUCTURE.

A plain, slow, float64 restatement of what the layer computes, written to be
checked by eye.  It shares no code with the CUDA library and never imports it.
Only the test suite, the smoke check and the CPU-baseline leg of the benchmark
may import it; the product path never routes through it.
"""
from .nvfp4_moe_oracle import *  # noqa: F401,F403
