"""CPU oracle for the MoE layer forward pass (test infrastructure only).

Only tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library.
"""
from .moe_oracle import *  # noqa: F401,F403
