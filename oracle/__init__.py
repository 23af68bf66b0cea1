"""CPU oracle for the slot-cached MoE layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.
"""
from .moe_oracle import *  # noqa: F401,F403
