"""Pins of the oracle's delayed-scaling state machine (CPU only).

The recipe is ``DelayedScaling(fp8_format=HYBRID, amax_history_len=16,
amax_compute_algo="max")`` (TE tutorial, code block 1); the state it keeps is
printed as ``scale`` and ``amax_history[0, :4]`` (TE tutorial, code block 4).
The closed form used here is written independently of the rolling buffer: the
scale after step t is fp8_max over the max of the amaxes of steps t-L+1..t.
"""
import math
import os

import numpy as np
import pytest

from oracle import fp8
from oracle.delayed_scaling import Recipe, ScalingState

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(fmt, L, amaxes):
    st = ScalingState(1, L)
    scales, invs = [], []
    for a in amaxes:
        st.record(0, np.float32(a))
        st.update([fmt])
        scales.append(float(st.scale[0]))
        invs.append(float(st.scale_inv[0]))
    return st, scales, invs


def _closed_form(fmt, L, amaxes):
    out, s = [], 1.0
    for t in range(len(amaxes)):
        window = amaxes[max(0, t - L + 1): t + 1]
        if any(math.isnan(w) for w in window):
            a = float("nan")
        else:
            a = max(window)
        if math.isfinite(a) and a > 0:
            cand = float(np.float32(fp8.FP8_MAX[fmt]) / np.float32(a))
            if math.isfinite(cand):
                s = cand
        out.append(s)
    return out


def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "delayed_scaling_sequences.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, L, am, exp = line.split()[:4]
            rows.append((fmt, int(L), [float(v) for v in am.split(",")], [float(v) for v in exp.split(",")]))
    return rows


@pytest.mark.parametrize("fmt,L,amaxes,expected", _golden())
def test_scripted_streams(fmt, L, amaxes, expected):
    _, scales, invs = _run(fmt, L, amaxes)
    assert scales == expected
    for s, i in zip(scales, invs):
        assert np.float32(i) == np.float32(np.float32(1.0) / np.float32(s))


@pytest.mark.parametrize("L", [1, 2, 3, 16, 1024])
@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_random_streams_follow_the_window_closed_form(L, fmt):
    rng = np.random.default_rng(L)
    am = list((np.exp(rng.standard_normal(60) * 3) * (rng.random(60) > 0.1)).astype(np.float32).astype(float))
    _, scales, _ = _run(fmt, L, am)
    assert scales == _closed_form(fmt, L, am)


def test_history_row_zero_is_the_latest_step_and_cur_is_cleared():
    st = ScalingState(2, 4)
    for t, (a, b) in enumerate([(1, 10), (2, 20), (3, 30)]):
        st.record(0, a)
        st.record(1, b)
        st.record(0, a / 2)  # a smaller amax in the same step does not lower it
        st.update([fp8.E4M3, fp8.E5M2])
    assert st.amax_history[:, 0].tolist() == [3, 2, 1, 0]
    assert st.amax_history[:, 1].tolist() == [30, 20, 10, 0]
    assert st.amax_cur.tolist() == [0, 0]
    assert st.scale[0] == np.float32(448 / 3) and st.scale[1] == np.float32(57344 / 30)


def test_first_step_casts_with_scale_one():
    st = ScalingState(4, 16)
    assert st.scale.tolist() == [1.0] * 4 and st.scale_inv.tolist() == [1.0] * 4


def test_tiny_amax_that_overflows_the_scale_keeps_it():
    _, scales, _ = _run(fp8.E5M2, 2, [1e-38, 0.5])
    assert scales == [1.0, 114688.0]


def test_resume_from_saved_state_equals_an_uninterrupted_run():
    rng = np.random.default_rng(11)
    am = rng.exponential(size=(40, 3)).astype(np.float32)
    fmts = [fp8.E4M3, fp8.E4M3, fp8.E5M2]
    a = ScalingState(3, 5)
    for t in range(40):
        for i in range(3):
            a.record(i, am[t, i])
        a.update(fmts)
    b = ScalingState(3, 5)
    for t in range(17):
        for i in range(3):
            b.record(i, am[t, i])
        b.update(fmts)
    c = b.copy()
    for t in range(17, 40):
        for i in range(3):
            c.record(i, am[t, i])
        c.update(fmts)
    for f in ("scale", "scale_inv", "amax_history", "amax_cur"):
        assert np.array_equal(getattr(a, f), getattr(c, f))


def test_recipe_formats():
    assert Recipe("hybrid").fwd_fmt() == fp8.E4M3 and Recipe("hybrid").bwd_fmt() == fp8.E5M2
    assert Recipe("e4m3").fwd_fmt() == fp8.E4M3 and Recipe("e4m3").bwd_fmt() == fp8.E4M3
    assert Recipe("e5m2").fwd_fmt() == fp8.E5M2 and Recipe("e5m2").bwd_fmt() == fp8.E5M2
