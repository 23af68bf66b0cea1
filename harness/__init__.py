"""Seeded synthetic workloads (configurations and input draws).

Shared by the oracle-side tests, the CUDA-side tests and the benchmark.  It
holds no MoE arithmetic: only shapes, seeds and random draws.
"""
from . import configs, gen  # noqa: F401
