"""Seeded synthetic workloads (shapes, sequence layouts, random tensors).

Shared by the oracle tests, the GPU parity tests and the bench; holds none of the
decoder's arithmetic.
"""
from .configs import (SLIDING, FULL, ModelShape, ImageSpan, Workload, CONFIGS,  # noqa: F401
                      cfg1, cfg2, cfg3, cfg4, cfg5, small_shape)
from .inputs import Inputs, f32_to_bf16_bits, bf16_bits_to_f32  # noqa: F401
