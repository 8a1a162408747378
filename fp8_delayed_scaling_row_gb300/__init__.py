"""GB300-native FP8 delayed-scaling LayerNormLinear / LayerNormMLP.

The compute path is liblnfp8.so (hand-written sm_103a CUDA behind a C ABI,
include/lnfp8.h); ``fp8_delayed_scaling_row_gb300.lnfp8`` is its Python
binding and loads the library on import (raising if it is not built).
``fp8_delayed_scaling_row_gb300.synth`` draws the seeded synthetic workloads.
"""
__all__ = ["lnfp8", "synth", "build"]
