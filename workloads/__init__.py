"""Seeded synthetic workloads (shapes, seeds and the planted input generator).

Shared by the oracle's tests, the GPU parity tests and the benchmark; it holds none of
the method's arithmetic.
"""
from .configs import WORKLOADS, Workload, get  # noqa: F401
