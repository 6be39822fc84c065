"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Holds the random draws and the quantization recipes of the workloads only: no
decode, no matrix product.
"""
from .configs import CONFIGS, make_dense, make_moe, zipf_route  # noqa: F401
