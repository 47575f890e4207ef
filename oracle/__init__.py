"""Plain float64 CPU oracle of the MoE layer forward (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
