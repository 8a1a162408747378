"""GELU between the two MLP GEMMs (oracle; test infrastructure only).

LayerNormMLP applies a GELU between its two linear layers (Turbo-charging guide,
"The building blocks: fused modules you'll use"; TE tutorial, code block 2,
whose plain-PyTorch block uses ``nn.GELU()``). The pages do not say which GELU;
the fused path uses the tanh approximation, and the exact erf form is kept here
behind ``approx="erf"`` because the tutorial's fallback block uses it.

Parity: pinned (gelu(0) = 0, gelu'(0) = 1/2, gelu(x) -> x for large x, agreement
with torch's gelu in fp64 for both forms, derivative against fp64 autograd).
"""
from __future__ import annotations

import math

import numpy as np

_K = math.sqrt(2.0 / math.pi)
_C = 0.044715


def gelu(h: np.ndarray, approx: str = "tanh") -> np.ndarray:
    """tanh form: 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3))); erf form: 0.5 h (1 + erf(h/sqrt 2))."""
    h = np.asarray(h, dtype=np.float64)
    if approx == "tanh":
        return 0.5 * h * (1.0 + np.tanh(_K * (h + _C * h ** 3)))
    if approx == "erf":
        from scipy.special import erf
        return 0.5 * h * (1.0 + erf(h / math.sqrt(2.0)))
    raise ValueError(approx)


def gelu_grad(h: np.ndarray, approx: str = "tanh") -> np.ndarray:
    """d gelu / d h, analytic."""
    h = np.asarray(h, dtype=np.float64)
    if approx == "tanh":
        t = np.tanh(_K * (h + _C * h ** 3))
        return 0.5 * (1.0 + t) + 0.5 * h * (1.0 - t * t) * _K * (1.0 + 3.0 * _C * h * h)
    if approx == "erf":
        from scipy.special import erf
        return 0.5 * (1.0 + erf(h / math.sqrt(2.0))) + h * np.exp(-0.5 * h * h) / math.sqrt(2.0 * math.pi)
    raise ValueError(approx)
