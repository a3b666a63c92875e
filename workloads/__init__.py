"""Seeded synthetic inputs for the eviction engine's five workloads.

This package holds input construction only (shapes, seeds, value
distributions); none of the eviction method's arithmetic.  Both the CUDA
path (tests, bench) and the oracle consume exactly the tensors it returns.
"""
from .generators import SHAPES, Shape, Workload, shape, scaled  # noqa: F401
