"""FP8 GEMM with per-tensor dequantisation and bf16 rounding (oracle; test
infrastructure only).

The linear layers run on "FP8 tensor cores" (TE tutorial, code block 1 prose),
taking the FP8 codes of both operands and undoing each operand's scale after the
product. With codes a, b and the inverse scales recorded when they were cast:

    C[i, j] = (sum_k dec(a[i, k]) * dec(b[j, k])) * (sinv_a * sinv_b) + bias[j]

The product sinv_a * sinv_b is formed first, in fp32 (the scales are fp32
state). The sum is taken in fp64 here (a library matmul of the exactly decoded
values), which is the exact result up to fp64 rounding; the GPU accumulates in
fp32 in another order, which the tolerance covers. Outputs handed on as bf16
tensors are rounded once, to nearest with ties to even.

Parity: pinned (small-integer FP8 inputs make every sum exact, so results equal
a brute-force triple loop and a fp64 matmul bit for bit; a transposed or swapped
operand, a dropped scale or bias fails those).
"""
from __future__ import annotations

import numpy as np

from .fp8 import decode


def dequant_scale(sinv_a, sinv_b) -> np.float32:
    return np.float32(np.float32(sinv_a) * np.float32(sinv_b))


def fp8_gemm(a_codes: np.ndarray, fmt_a: str, b_codes: np.ndarray, fmt_b: str,
             sinv_a, sinv_b, bias: np.ndarray | None = None) -> np.ndarray:
    """C = (dec(A) @ dec(B)^T) * (sinv_a * sinv_b) + bias, in fp64.

    a_codes: [M, K] codes, b_codes: [N, K] codes (both indexed [row, k], the
    ``nn.Linear`` [out, in] convention for B)."""
    a = decode(a_codes, fmt_a)
    b = decode(b_codes, fmt_b)
    acc = a @ b.T
    out = acc * np.float64(dequant_scale(sinv_a, sinv_b))
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)[None, :]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round values to bf16 (nearest, ties to even) via fp32; return uint16 bits.

    The fp64 value is first rounded to fp32 (nearest), then the low 16 bits of
    the fp32 pattern are rounded off with ties to even; NaN stays a quiet NaN."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    keep_even = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_even) >> np.uint64(16)).astype(np.uint16)
    r = np.where(np.isnan(f), np.uint16(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
