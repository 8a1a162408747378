"""Delayed-scaling recipe and its per-tensor state machine (oracle; test
infrastructure only).

The recipe (TE tutorial, code block 1; Turbo-charging guide, "Playing with
lower-precision formats: BF16 vs FP8") is ``DelayedScaling(fp8_format=HYBRID,
amax_history_len=16, amax_compute_algo="max")``: each FP8 tensor keeps a
rolling history of its recent amaxes, and the scale used to cast it is derived
from that history rather than from the tensor being cast ("delayed"). The
tutorial's state dump (code block 4) prints ``scale`` (one entry per FP8 tensor)
and ``amax_history[0, :4]`` (history index first; row 0 is the most recent).

State per tensor slot i (all fp32):
  scale[i], scale_inv[i], amax_history[L][i], amax_cur[i] (running step).
Initial: scale = scale_inv = 1, history = 0, cur = 0.
During a step: every cast of tensor i uses scale[i]; cur[i] = max(cur[i], amax).
At the update after the step:
  1. history rows move down one: history[j] = history[j-1] for j = L-1 .. 1;
  2. history[0] = cur, then cur = 0;
  3. a = max over the L rows ("max" is the only algorithm the pages name);
  4. if a is finite and > 0 and s = fp8_max / a (one fp32 division, margin 0)
     is finite, scale = s and scale_inv = 1 / s (fp32); otherwise both keep
     their value.
So step 1 casts with scale 1 and step t+1 uses the amaxes of steps
max(1, t-L+1) .. t. Readings (not on the pages): fp8_max is 448 for E4M3 and
57344 for E5M2, margin 0, and a zero / non-finite window keeps the old scale.

HYBRID maps forward tensors (LayerNorm output, weights, GELU output) to E4M3 and
gradients (dY, dH) to E5M2; the E4M3 format uses E4M3 for all of them; E5M2
uses E5M2 for all of them.

Parity: pinned (scripted amax streams against the closed form
scale_t = fp8_max / max(amax over the last L steps), keep-on-zero / NaN cases,
resume-from-saved-state equals an uninterrupted run).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .fp8 import E4M3, E5M2, FP8_MAX

HYBRID = "hybrid"
FORMAT_E4M3 = "e4m3"
FORMAT_E5M2 = "e5m2"


@dataclass
class Recipe:
    fp8_format: str = HYBRID
    amax_history_len: int = 16
    amax_compute_algo: str = "max"
    margin: int = 0

    def fwd_fmt(self) -> str:
        return E5M2 if self.fp8_format == FORMAT_E5M2 else E4M3

    def bwd_fmt(self) -> str:
        return E4M3 if self.fp8_format == FORMAT_E4M3 else E5M2


def _bits(x) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0] & 0x7FFFFFFF)


def _from_bits(u: int) -> np.float32:
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


class ScalingState:
    """The delayed-scaling state of n FP8 tensors (the ``fp8_meta`` of one module
    direction, e.g. ``scaling_fwd``)."""

    def __init__(self, n: int, history_len: int):
        if history_len < 1:
            raise ValueError("amax_history_len must be >= 1")
        self.n = n
        self.L = history_len
        self.scale = np.ones(n, dtype=np.float32)
        self.scale_inv = np.ones(n, dtype=np.float32)
        self.amax_history = np.zeros((history_len, n), dtype=np.float32)
        self.amax_cur = np.zeros(n, dtype=np.float32)

    def copy(self) -> "ScalingState":
        s = ScalingState(self.n, self.L)
        s.scale[:] = self.scale
        s.scale_inv[:] = self.scale_inv
        s.amax_history[:] = self.amax_history
        s.amax_cur[:] = self.amax_cur
        return s

    def record(self, i: int, amax_value) -> None:
        """cur[i] = max(cur[i], amax) in the fp32 magnitude bit order."""
        self.amax_cur[i] = _from_bits(max(_bits(self.amax_cur[i]), _bits(amax_value)))

    def update(self, fmts: list[str], algo: str = "max", margin: int = 0) -> None:
        """The end-of-step update, steps 1-4 above, for every slot."""
        if algo != "max":
            raise ValueError("only amax_compute_algo='max' is defined by the pages")
        for i in range(self.n):
            for j in range(self.L - 1, 0, -1):
                self.amax_history[j, i] = self.amax_history[j - 1, i]
            self.amax_history[0, i] = self.amax_cur[i]
            self.amax_cur[i] = np.float32(0.0)
            a = _from_bits(max(_bits(v) for v in self.amax_history[:, i]))
            if np.isfinite(a) and a > 0:
                s = np.float32(np.float32(FP8_MAX[fmts[i]]) / a)
                if margin:
                    s = np.float32(s / np.float32(2.0 ** margin))
                if np.isfinite(s):
                    self.scale[i] = s
                    self.scale_inv[i] = np.float32(np.float32(1.0) / s)
