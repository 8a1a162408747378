"""Seeded synthetic inputs for the FP8 delayed-scaling LayerNormLinear /
LayerNormMLP workloads.

This module is the one piece shared by the CPU oracle, the CUDA path's tests and
the benchmark. It draws input tensors only and holds none of the method's
arithmetic (no LayerNorm, no FP8 cast, no GEMM, no scaling).

Every tensor comes from numpy's counter-based Philox generator keyed by
(seed, step, tensor id), so the same call gives the same bytes on any machine.
The base seed 1234 is the tutorial's own ``torch.manual_seed(1234)``
(TE tutorial, code block 1). bf16 tensors are returned as ``uint16`` bit
patterns; fp32 tensors as ``float32``.

Distributions follow the workloads' descriptions:
  * activations X ~ N(0, 1), optionally with each entry independently scaled
    x50 with probability 0.001 ("0.1% outliers"), or drawn from a Student-t
    with 3 degrees of freedom (heavy tails);
  * LayerNorm gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1);
  * weights ~ N(0, 0.02) (0.02 is a standard deviation);
  * upstream gradient dY ~ N(0, 0.01).
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 1234

# Tensor ids keep the streams of different tensors of one step apart.
TID = {
    "x": 1, "gamma": 2, "beta": 3, "w": 4, "b": 5, "w1": 6, "b1": 7, "w2": 8,
    "b2": 9, "dy": 10, "attn": 11, "outlier": 12, "chi": 13, "gamma2": 14,
    "beta2": 15, "wqkv": 16, "bqkv": 17, "wproj": 18, "bproj": 19,
}


def _gen(seed: int, step: int, tid: int, layer: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), int(step), int(tid), int(layer)])
    return np.random.Generator(np.random.Philox(ss))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (nearest, ties to even) and return the bits.

    Only used to store generated samples in the bf16 input format."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(shape, std: float, seed: int, step: int, tid: int, layer: int = 0) -> np.ndarray:
    g = _gen(seed, step, tid, layer)
    return (g.standard_normal(size=shape, dtype=np.float64) * std).astype(np.float32)


def activations(rows: int, cols: int, *, dist: str = "normal", seed: int = BASE_SEED,
                step: int = 0, tid: int = TID["x"], layer: int = 0) -> np.ndarray:
    """bf16 bits of an activation tensor [rows, cols].

    dist: "normal"   N(0,1)
          "outliers" N(0,1), each entry x50 with probability 0.001
          "t3"       Student-t, 3 degrees of freedom: N / sqrt(chi2_3 / 3)
    """
    g = _gen(seed, step, tid, layer)
    z = g.standard_normal(size=(rows, cols), dtype=np.float64)
    if dist == "normal":
        pass
    elif dist == "outliers":
        hit = g.random(size=(rows, cols)) < 1e-3
        z = np.where(hit, z * 50.0, z)
    elif dist == "t3":
        chi2 = (g.standard_normal(size=(3, rows, cols), dtype=np.float64) ** 2).sum(axis=0)
        z = z / np.sqrt(chi2 / 3.0)
    else:
        raise ValueError(f"unknown activation distribution {dist!r}")
    return f32_to_bf16_bits(z.astype(np.float32))


def ln_params(d: int, *, seed: int = BASE_SEED, layer: int = 0, which: int = 0):
    """(gamma, beta) bf16 bits, gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1)."""
    tg, tb = (TID["gamma"], TID["beta"]) if which == 0 else (TID["gamma2"], TID["beta2"])
    gamma = 1.0 + normal((d,), 0.1, seed, 0, tg, layer)
    beta = normal((d,), 0.1, seed, 0, tb, layer)
    return f32_to_bf16_bits(gamma), f32_to_bf16_bits(beta)


def weight(n_out: int, n_in: int, *, std: float = 0.02, seed: int = BASE_SEED,
           tid: int = TID["w"], layer: int = 0) -> np.ndarray:
    """bf16 bits of a weight [out, in] (the nn.Linear layout) ~ N(0, std)."""
    return f32_to_bf16_bits(normal((n_out, n_in), std, seed, 0, tid, layer))


def bias(n: int, *, std: float = 0.0, seed: int = BASE_SEED, tid: int = TID["b"],
         layer: int = 0) -> np.ndarray:
    """bf16 bits of a bias [n]; std 0 gives the all-zero bias of the workloads."""
    if std == 0.0:
        return np.zeros((n,), dtype=np.uint16)
    return f32_to_bf16_bits(normal((n,), std, seed, 0, tid, layer))


def grad(rows: int, cols: int, *, std: float = 0.01, seed: int = BASE_SEED, step: int = 0,
         tid: int = TID["dy"], layer: int = 0) -> np.ndarray:
    """bf16 bits of an upstream gradient [rows, cols] ~ N(0, std)."""
    return f32_to_bf16_bits(normal((rows, cols), std, seed, step, tid, layer))


def mlp_params(d: int, f: int, *, seed: int = BASE_SEED, layer: int = 0, bias_std: float = 0.0):
    """gamma, beta, W1 [f,d], b1 [f], W2 [d,f], b2 [d] for one LayerNormMLP."""
    gamma, beta = ln_params(d, seed=seed, layer=layer, which=1)
    w1 = weight(f, d, seed=seed, tid=TID["w1"], layer=layer)
    w2 = weight(d, f, seed=seed, tid=TID["w2"], layer=layer)
    b1 = bias(f, std=bias_std, seed=seed, tid=TID["b1"], layer=layer)
    b2 = bias(d, std=bias_std, seed=seed, tid=TID["b2"], layer=layer)
    return dict(gamma=gamma, beta=beta, w1=w1, b1=b1, w2=w2, b2=b2)


def linear_params(n_out: int, n_in: int, *, seed: int = BASE_SEED, layer: int = 0,
                  ln: bool = True, bias_std: float = 0.0, wtid: int = TID["w"],
                  btid: int = TID["b"]):
    """(gamma, beta or None), W [n_out, n_in], b [n_out] for one LayerNormLinear / Linear."""
    p = dict(w=weight(n_out, n_in, seed=seed, tid=wtid, layer=layer),
             b=bias(n_out, std=bias_std, seed=seed, tid=btid, layer=layer))
    if ln:
        p["gamma"], p["beta"] = ln_params(n_in, seed=seed, layer=layer, which=0)
    else:
        p["gamma"], p["beta"] = None, None
    return p
