"""Seeded synthetic inputs shared by the CUDA path, its tests and the oracle.

This package produces input bytes only: planted-spectrum activations and
output gradients, weights, GELU activations and the Givens drift of a planted
subspace.  It holds none of the low-rank backward's arithmetic, so that the
oracle and the CUDA library can both consume the same bytes without sharing
any code of the method.
"""

from .gen import (  # noqa: F401
    WORKLOADS,
    LayerInputs,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    gelu_activations,
    givens_rotate,
    planted_batch,
    planted_basis,
    sigma_profile,
    seed_for,
    weight,
    workload,
)
