"""Pins of the oracle's FP8 codec, scaled cast and amax (CPU only).

The codec is fixed by the OCP 8-bit floating point specification, which the
pages name only as "E4M3" / "E5M2" (TE tutorial, code block 1 recipe; the
Turbo-charging guide, "Playing with lower-precision formats: BF16 vs FP8").
"""
import math
import os
import struct

import numpy as np
import pytest

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_decode_tables_have_the_spec_landmarks():
    e4 = fp8.decode(np.arange(256), fp8.E4M3)
    e5 = fp8.decode(np.arange(256), fp8.E5M2)
    # NaN / Inf counts: E4M3 has only S.1111.111 as NaN and no Inf;
    # E5M2 has 2 Inf and 6 NaN codes.
    assert np.isnan(e4).sum() == 2 and np.isinf(e4).sum() == 0
    assert np.isnan(e5).sum() == 6 and np.isinf(e5).sum() == 2
    assert np.nanmax(e4) == 448.0 and np.nanmin(e4) == -448.0
    assert np.nanmax(e5[np.isfinite(e5)]) == 57344.0
    pos4 = e4[1:0x7F]
    pos5 = e5[1:0x7C]
    assert pos4.min() == 2.0 ** -9 and pos5.min() == 2.0 ** -16
    assert fp8.decode_code(0x08, fp8.E4M3) == 2.0 ** -6
    assert fp8.decode_code(0x04, fp8.E5M2) == 2.0 ** -14
    # positive codes are strictly increasing in value; negative codes mirror them
    assert np.all(np.diff(e4[:0x7F]) > 0) and np.all(np.diff(e5[:0x7C]) > 0)
    assert np.array_equal(e4[0x80:0xFF], -e4[:0x7F])
    assert np.array_equal(e5[0x80:0xFC], -e5[:0x7C])
    # E4M3 carries 3 mantissa bits: between 1 and 2 the spacing is 1/8; E5M2: 1/4
    assert np.allclose(np.diff(e4[0x38:0x41]), 0.125)
    assert np.allclose(np.diff(e5[0x3C:0x41]), 0.25)


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_every_code_round_trips(fmt):
    codes = np.arange(256)
    vals = fp8.decode(codes, fmt)
    finite = np.isfinite(vals)
    back = fp8.encode(vals[finite].astype(np.float32), fmt)
    assert np.array_equal(back, codes[finite].astype(np.uint8))
    nan = np.isnan(vals)
    assert np.all(np.isnan(fp8.decode(fp8.encode(vals[nan].astype(np.float32), fmt), fmt)))


def _golden_cases():
    out = []
    with open(os.path.join(GOLDEN, "fp8_cast_cases.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, val, code = line.split()[:3]
            out.append((fmt, float(val), int(code, 16), line))
    return out


@pytest.mark.parametrize("fmt,val,code,line", _golden_cases())
def test_hand_worked_cast_cases(fmt, val, code, line):
    got = int(fp8.encode(np.array([val], dtype=np.float32), fmt)[0])
    assert got == code, f"{line}: got 0x{got:02X}"


def _boundary_points(fmt):
    """Every decision point of the encoder: each representable magnitude, each
    midpoint between neighbours, and the fp32 values on either side of it."""
    vals = fp8.decode(np.arange(128), fmt)
    vals = vals[np.isfinite(vals)]
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(0))
    pts = np.concatenate([pts, up, dn])
    return np.concatenate([pts, -pts])


@pytest.mark.parametrize("fmt,tdt", [(fp8.E4M3, "float8_e4m3fn"), (fp8.E5M2, "float8_e5m2")])
def test_encoder_matches_torch_float8_on_every_boundary(fmt, tdt):
    torch = pytest.importorskip("torch")
    dt = getattr(torch, tdt, None)
    if dt is None:
        pytest.skip("this torch has no float8 dtypes")
    rng = np.random.default_rng(7)
    rand = (rng.standard_normal(200_000) * np.exp2(rng.integers(-20, 20, 200_000))).astype(np.float32)
    x = np.concatenate([_boundary_points(fmt), rand]).astype(np.float32)
    mx = fp8.FP8_MAX[fmt]
    # torch's cast is round-to-nearest-even but not saturating: clamp first.
    t = torch.from_numpy(np.clip(x, -mx, mx)).to(dt).view(torch.uint8).numpy()
    ours = fp8.encode(x, fmt)
    # torch maps a zero result of a negative input to 0x80 as well
    assert np.array_equal(ours, t), np.nonzero(ours != t)[0][:10]


def test_saturation_and_nan_policy():
    x = np.array([np.inf, -np.inf, 1e30, -1e30, np.nan], dtype=np.float32)
    e4 = fp8.encode(x, fp8.E4M3)
    assert list(e4[:4]) == [0x7E, 0xFE, 0x7E, 0xFE]
    assert np.isnan(fp8.decode(e4[4:], fp8.E4M3)).all()
    e5 = fp8.encode(x, fp8.E5M2)
    assert list(e5[:4]) == [0x7B, 0xFB, 0x7B, 0xFB]
    assert np.isnan(fp8.decode(e5[4:], fp8.E5M2)).all()


def test_quantize_is_one_fp32_multiply_then_the_cast():
    # 1 + 2^-23 times 1 + 2^-23 is 1 + 2^-22 + 2^-46; in fp32 the product rounds
    # to 1 + 2^-22, which E4M3 rounds to 1.0. A power-of-two scale is exact.
    x = np.array([f32(1 + 2 ** -23)], dtype=np.float32)
    assert fp8.scale_mul(x, np.float32(1 + 2 ** -23))[0] == np.float32(1 + 2 ** -22)
    assert fp8.quantize(x, np.float32(1 + 2 ** -23), fp8.E4M3)[0] == 0x38
    # scale 2^k only moves the exponent: 3.0 * 64 = 192 = 1.5 * 2^7 -> e=14, m=4
    assert fp8.quantize(np.array([3.0], np.float32), 64.0, fp8.E4M3)[0] == 0x74
    # a scale that pushes past the max saturates
    assert fp8.quantize(np.array([2.0], np.float32), 448.0, fp8.E4M3)[0] == 0x7E


def test_amax_is_the_max_magnitude_in_bit_order():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((37, 53)) * 10).astype(np.float32)
    assert fp8.amax(x) == max(abs(float(v)) for v in x.ravel())
    assert fp8.amax(np.zeros((0, 4), np.float32)) == 0.0
    y = x.copy()
    y[3, 4] = -np.inf
    assert fp8.amax(y) == np.inf
    y[5, 6] = np.nan
    assert math.isnan(fp8.amax(y))
    assert fp8.amax(np.array([-0.0, 0.0], np.float32)) == 0.0
