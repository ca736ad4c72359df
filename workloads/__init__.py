"""Seeded synthetic inputs for the verification path.

This package is shared by the GPU tests, the benchmark and the oracle's tests. It draws random
numbers and lays them out; it holds none of the verification arithmetic.
"""
from .configs import CONFIGS, Config, get_config  # noqa: F401
from .generate import (Workload, bf16_bits_to_f32, bf16_round, filter_params,  # noqa: F401
                       make_workload)
