"""Seeded synthetic inputs for the Flint MoE layer (host numpy + CUDA generator).

Shared by the tests, the benchmark and the oracle's callers; it holds none of
the layer's arithmetic.
"""
from . import gen  # noqa: F401
