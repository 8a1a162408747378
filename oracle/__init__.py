"""CPU oracle for the FP8 delayed-scaling LayerNormLinear / LayerNormMLP step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only the tests, the smoke check and the benchmark's
CPU-baseline leg use it. It shares no code with the CUDA library, and the
library never calls it (a missing CUDA extension is an error, never a reason
to fall back to the CPU).

It is a plain, slow, step-by-step restatement of what the method computes, in
numpy, in the order the pages describe it. Floating point is fp64 except where
the method itself fixes a precision: the FP8 cast takes an fp32 value times an
fp32 scale, the amax is taken over those fp32 values, and the scale arithmetic
of delayed scaling is fp32. Where the pages leave a step open, the reading
taken is stated in the function's docstring.

Sources (cited by title and section):
  * "Accelerating Transformer Training with NVIDIA Transformer Engine, Fused
    Kernels, BF16, FP8, and GPU Benchmarking" (the TE tutorial), code blocks 1-5;
  * "Turbo-charging your transformer training: a hands-on guide" (the
    Turbo-charging guide), by section heading;
  * the OCP 8-bit floating point specification (OFP8) for the E4M3 / E5M2 bit
    layouts, which the pages name but do not spell out.

Parity status per function: see each module's header. Functions whose result
with quantisation switched on has no independent pin say "parity unpinned".
"""
from . import fp8, layernorm, gelu, gemm, delayed_scaling, modules  # noqa: F401
