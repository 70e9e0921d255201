"""CPU oracle of the MoE expert block (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU baseline and
reference arm may import this package; the CUDA library never does.
"""
from .moe_oracle import *  # noqa: F401,F403
