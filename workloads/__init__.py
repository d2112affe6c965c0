"""Seeded synthetic workloads (shapes, seeds and input generators).

This package is shared by the CUDA path's tests and bench and by the oracle.
It holds none of the sparse-attention method's arithmetic.
"""
from .configs import WORKLOADS, Workload, scaled, workload  # noqa: F401
