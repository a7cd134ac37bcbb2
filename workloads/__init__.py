"""Seeded synthetic inputs for GPTQ layer quantization.

This package only draws random numbers.  It holds none of the method's arithmetic, so
both the CUDA path (through its tests and the bench) and the float64 oracle can take
their inputs from it.
"""

from .synthetic import (  # noqa: F401
    CONFIGS,
    LayerConfig,
    channel_multipliers,
    make_permutation,
    make_upper_factor,
    make_weight,
    make_tokens,
    make_tokens_chunk,
    token_chunks,
)
