"""Plain CPU oracle of the MoE layer (test infrastructure only): C++ loops in moe_oracle.cpp,
reached through the ctypes wrapper moe_oracle.py.

Only the tests, the smoke check and the benchmark's CPU legs use it.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
