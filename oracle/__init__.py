"""Test-only CPU oracle (float64 numpy) for the MC-Sparse hot path.

Imported only by tests/, the package smoke check and the benchmark's CPU
baseline; the product path never calls it.
"""
from .mcs_oracle import *  # noqa: F401,F403
