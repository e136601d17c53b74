"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the bench.

Holds shapes, seeds and input generation only; no arithmetic of the method.
"""
from .configs import CONFIGS, ORDER, LocksWorkload, get  # noqa: F401
from .generator import (LocksInputs, bf16_bits_to_f32, f32_to_bf16_bits,  # noqa: F401
                        generate)
