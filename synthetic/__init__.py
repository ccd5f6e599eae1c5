"""Seeded synthetic inputs (weights W, calibration activations X) for GPTQ layers.

This module is the only code shared by the oracle and the CUDA path: it draws
numbers and rounds them to the storage dtype.  It holds none of the
quantization arithmetic.
"""
from .layers import (  # noqa: F401
    CHUNK_ROWS,
    LAYERS,
    LayerSpec,
    TensorSpec,
    bf16_bits_to_f32,
    custom_layer,
    generate,
    generate_rows,
    outlier_channels,
)
