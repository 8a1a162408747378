"""Row LayerNorm forward and backward (oracle; test infrastructure only).

The fused modules start with a LayerNorm over each token row
(TE tutorial, code block 1: ``te.LayerNorm(H)``, ``te.LayerNormLinear(H, 3*H)``,
``te.LayerNormMLP(H, 4*H)``; Turbo-charging guide, "The building blocks: fused
modules you'll use": LayerNormLinear "combines layer-norm and a linear mapping",
LayerNormMLP bundles "layer-norm, two linear layers, GELU").

The pages print no formula. This is the textbook LayerNorm with the biased
variance and eps = 1e-5 (the PyTorch/TE default), statistics in fp64, output
stored as fp32 (the value the FP8 cast consumes). The backward is its exact
derivative.

Parity: pinned (zero mean and var/(var+eps) variance before the affine, a
constant row maps to beta, agreement with torch.layer_norm in fp64, backward
against fp64 autograd and central finite differences).
"""
from __future__ import annotations

import numpy as np

EPS = 1e-5


def forward(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = EPS):
    """y = (x - mu) * rsigma * gamma + beta per row.

    x: [M, D] values (any float dtype); gamma, beta: [D].
    Returns (y fp32 [M, D], mu fp32 [M], rsigma fp32 [M]) where
    mu = sum(x)/D, var = sum((x - mu)^2)/D, rsigma = 1/sqrt(var + eps)."""
    xd = np.asarray(x, dtype=np.float64)
    d = xd.shape[1]
    mu = xd.sum(axis=1) / d
    xc = xd - mu[:, None]
    var = (xc * xc).sum(axis=1) / d
    rsigma = 1.0 / np.sqrt(var + eps)
    y = xc * rsigma[:, None] * np.asarray(gamma, np.float64)[None, :] + np.asarray(beta, np.float64)[None, :]
    return y.astype(np.float32), mu.astype(np.float32), rsigma.astype(np.float32)


def backward(dy: np.ndarray, x: np.ndarray, gamma: np.ndarray, eps: float = EPS):
    """Gradients of LayerNorm with respect to x, gamma and beta (fp64).

    With xhat = (x - mu) * rsigma and g = dy * gamma (per element):
      dx     = rsigma * (g - mean_row(g) - xhat * mean_row(g * xhat))
      dgamma = sum_rows(dy * xhat)
      dbeta  = sum_rows(dy)
    Statistics are recomputed here in fp64 from x."""
    xd = np.asarray(x, dtype=np.float64)
    dyd = np.asarray(dy, dtype=np.float64)
    d = xd.shape[1]
    mu = xd.sum(axis=1) / d
    xc = xd - mu[:, None]
    var = (xc * xc).sum(axis=1) / d
    rsigma = 1.0 / np.sqrt(var + eps)
    xhat = xc * rsigma[:, None]
    g = dyd * np.asarray(gamma, np.float64)[None, :]
    dx = rsigma[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    dgamma = (dyd * xhat).sum(axis=0)
    dbeta = dyd.sum(axis=0)
    return dx, dgamma, dbeta
