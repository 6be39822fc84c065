"""CPU oracle of the fused-dequant quantized GEMM.  Test infrastructure only:
imported by the tests, the smoke check and the benchmark's CPU-baseline leg."""
from .hq_oracle import *  # noqa: F401,F403
