"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This package holds no arithmetic of the method: it only draws random tensors
(activations, raw weights before any quantization, adapter tables, per-token
adapter indices and the prefill mask) with the shapes and value laws of the
workloads, and rounds them to bf16 where the layer takes bf16 inputs.
"""
from .inputs import (  # noqa: F401
    LLAMA8B_PROJECTIONS,
    LLAMA70B_PROJECTIONS,
    ProjectionInputs,
    make_projection,
    zipf_indices,
)
