"""Seeded synthetic inputs shared by the oracle and the CUDA library's tests and bench.

This package holds data generation only (counter-based normal streams, bf16
rounding of activations, per-128x128-block e4m3 quantisation of weights); none
of the layer's arithmetic.
"""
from .configs import FAMILIES, Family, family, parse_workload, workload_name  # noqa: F401
from .synth import (LayerWeights, LayerWeightsFP4, bf16_bits_to_f32, blockwise_e4m3,  # noqa: F401
                    e4m3_encode, make_weights, make_weights_fp4, make_x, normal_bf16, normal_f32,
                    nvfp4)
