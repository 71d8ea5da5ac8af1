"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA side.

Holds random-number generation and input arrangement only; none of the
method's arithmetic lives here.
"""
from . import rng, workload  # noqa: F401
from .workload import BLOCK, WORKLOADS, Workload  # noqa: F401
