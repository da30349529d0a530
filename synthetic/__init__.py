"""Seeded synthetic inputs for the VLA forward recurrence.

This package produces input tensors only. It holds none of the method's
arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA path can take
their inputs from it without sharing any computation.
"""

from .generator import (  # noqa: F401
    CONFIGS,
    VLAInputs,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_config,
    make_inputs,
    make_recall_stream,
    normals,
    uniforms,
)
