"""Seeded synthetic workloads (shapes, sequence layouts, random tensors).

Shared by the oracle tests, the GPU parity tests and the bench; holds none of the
decoder's arithmetic.
"""
from .configs import (SLIDING, FULL, ModelShape, ImageSpan, Workload, WORKLOADS,  # noqa: F401
                      layer_fp32_T128, pair_T2048, stack28_T8192, decode_B64_cache4096, varlen_T32768, small_shape)
from .inputs import Inputs, f32_to_bf16_bits, bf16_bits_to_f32  # noqa: F401
