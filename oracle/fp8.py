"""FP8 codec, scaled cast and amax (oracle; test infrastructure only).

What the method needs from FP8: two 8-bit formats, E4M3 for forward tensors and
E5M2 for gradients under the HYBRID recipe (TE tutorial, code block 1: the FP8
recipe with ``recipe.Format.HYBRID``; Turbo-charging guide, "Playing with
lower-precision formats: BF16 vs FP8": HYBRID "mixes E4M3 and E5M2"). The pages
give no bit layout, maximum or rounding rule; this module takes them from the
OCP 8-bit floating point specification:

  E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits. No infinities;
               S.1111.111 is NaN, so the largest finite value is 1.75 * 2^8 = 448.
  E5M2:        1 sign, 5 exponent (bias 15), 2 mantissa bits. IEEE-like:
               exponent 31 with mantissa 0 is Inf, else NaN; max 1.75 * 2^15 = 57344.

The cast rounds an fp32 value to the nearest representable value with ties to
the even code and saturates: magnitudes at or beyond the largest finite value
(Inf included) become +-max; NaN stays NaN.

Parity: pinned (exhaustive 256-code decode/round-trip, hand-worked cases at and
beyond saturation, an independent cross-check against torch's float8 casts over
every rounding boundary).
"""
from __future__ import annotations

import numpy as np

E4M3 = "e4m3"
E5M2 = "e5m2"

FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}
_BITS = {E4M3: (4, 3, 7), E5M2: (5, 2, 15)}  # exponent bits, mantissa bits, bias


def decode_code(code: int, fmt: str) -> float:
    """Value of one FP8 code, straight from the bit-layout definition."""
    ebits, mbits, bias = _BITS[fmt]
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    emax = (1 << ebits) - 1
    if fmt == E4M3 and e == emax and m == (1 << mbits) - 1:
        return float("nan")
    if fmt == E5M2 and e == emax:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:  # subnormal: no implicit one, exponent 1 - bias
        return sign * (m / (1 << mbits)) * 2.0 ** (1 - bias)
    return sign * (1.0 + m / (1 << mbits)) * 2.0 ** (e - bias)


_TABLE = {f: np.array([decode_code(c, f) for c in range(256)], dtype=np.float64) for f in (E4M3, E5M2)}


def decode(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Exact fp64 value of every code in ``codes`` (uint8 array)."""
    return _TABLE[fmt][np.asarray(codes, dtype=np.uint8)]


def _positive_finite(fmt: str):
    """Codes 0..max_code and their values; positive codes are monotonic in value."""
    t = _TABLE[fmt][:128]
    max_code = int(np.nonzero(np.isfinite(t))[0].max())
    return np.arange(max_code + 1), t[: max_code + 1]


def encode(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round fp32 values to FP8 codes: nearest, ties to even code, saturating.

    The nearest representable value is found by searching the sorted table of
    non-negative finite values; on an exact tie the code with the even last bit
    (the even mantissa) wins. |x| >= max (including Inf) gives the max code.
    NaN gives the all-ones code with the input's sign (0x7F / 0xFF)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    neg = np.signbit(x)
    codes, vals = _positive_finite(fmt)
    vmax = vals[-1]
    i = np.clip(np.searchsorted(vals, a, side="left"), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    # 2a vs lo + hi decides the nearer neighbour exactly (all terms are dyadic
    # with few significant bits, so the fp64 sums below are exact).
    two_a = 2.0 * a
    mid = lo + hi
    pick_hi = (two_a > mid) | ((two_a == mid) & ((codes[i] & 1) == 0))
    out = np.where(pick_hi, codes[i], codes[i - 1]).astype(np.int64)
    out = np.where(a == 0.0, 0, out)
    out = np.where(a >= vmax, codes[-1], out)  # saturate, Inf included
    out = np.where(neg, out | 0x80, out)
    out = np.where(np.isnan(x), np.where(neg, 0xFF, 0x7F), out)
    return out.astype(np.uint8)


def scale_mul(x: np.ndarray, scale) -> np.ndarray:
    """fp32 x times fp32 scale, one IEEE round-to-nearest multiply."""
    return (np.asarray(x, dtype=np.float32) * np.float32(scale)).astype(np.float32)


def quantize(x: np.ndarray, scale, fmt: str) -> np.ndarray:
    """The scaled cast of delayed scaling: code = encode(fp32(x) * scale).

    Reading: the tracked scale multiplies the tensor before the cast (so
    scale_inv = 1/scale undoes it after the GEMM); the pages say only that the
    recipe "rescales" each tensor using its amax (Turbo-charging guide,
    "Playing with lower-precision formats: BF16 vs FP8")."""
    return encode(scale_mul(x, scale), fmt)


def amax(x: np.ndarray) -> np.float32:
    """Maximum absolute value of a tensor of fp32 values, NaN-propagating.

    "tracks the maximum absolute value (amax) of each tensor" (Turbo-charging
    guide, "Playing with lower-precision formats: BF16 vs FP8"). Magnitudes are
    ordered by their fp32 bit patterns (sign cleared), so NaN > Inf > finite and
    the result of an empty tensor is 0."""
    x = np.asarray(x, dtype=np.float32)
    if x.size == 0:
        return np.float32(0.0)
    bits = (x.view(np.uint32) & np.uint32(0x7FFFFFFF)).max()
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def max_bits(a, b) -> np.float32:
    """max of two non-negative fp32 magnitudes in the same bit order as amax."""
    ua = np.array([a], dtype=np.float32).view(np.uint32)[0] & 0x7FFFFFFF
    ub = np.array([b], dtype=np.float32).view(np.uint32)[0] & 0x7FFFFFFF
    return np.array([max(ua, ub)], dtype=np.uint32).view(np.float32)[0]
