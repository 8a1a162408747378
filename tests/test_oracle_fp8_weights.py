"""Pins of the oracle's module variants. FP8-stored weights (fp8_model_init, TE
tutorial closing list): the one-time conversion against what the FP8 formats
fix, and the modules' FP8-weight branch against the bf16-weight branch and the
exact fp64 layer. The residual add ahead of a LayerNorm module: against torch's
own bf16 addition, and a zero residual against no residual."""
import os

import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8, modules as omod
from oracle.delayed_scaling import Recipe, ScalingState
from oracle.gemm import bf16_to_f32

# mantissa bits and the smallest normal exponent of each format
FMT = {fp8.E4M3: (3, -6), fp8.E5M2: (2, -14)}


def _weight(rows, cols, seed=0):
    return synth.linear_params(rows, cols, ln=False, layer=seed, bias_std=0.0)["w"]


@pytest.mark.parametrize("fmt_name,margin", [("hybrid", 0), ("e5m2", 0), ("hybrid", 3), ("e4m3", 1)])
def test_quantize_weight_bounds(fmt_name, margin):
    rec = Recipe(fmt_name, 16, margin=margin)
    fmt = rec.fwd_fmt()
    w = _weight(96, 64)
    W = bf16_to_f32(w).astype(np.float64)
    codes, sinv, st = omod.quantize_weight(w, rec)
    dec = fp8.decode(codes, fmt).astype(np.float64)
    # the largest |w| lands exactly on fp8_max / 2^margin (the scale is fp8_max / amax / 2^margin)
    assert np.abs(dec).max() == fp8.FP8_MAX[fmt] / 2.0 ** margin
    assert np.sign(dec[np.unravel_index(np.abs(W).argmax(), W.shape)]) == np.sign(W.flat[np.abs(W).argmax()])
    # every element within half a unit in the last place of its FP8 value (normals: relative,
    # subnormals: half the subnormal spacing), plus the fp32 rounding of the scale
    m, emin = FMT[fmt]
    scale = np.float64(st.scale[0])
    v = W * scale
    half_ulp = np.where(np.abs(v) >= 2.0 ** emin, np.abs(v) * 2.0 ** -(m + 1), 2.0 ** (emin - m - 1))
    assert np.all(np.abs(dec - v) <= half_ulp * (1 + 1e-6) + np.abs(v) * 2 ** -22)
    # scale_inv is the fp32 reciprocal of the scale; the state holds the amax in history row 0
    assert sinv == np.float32(np.float32(1.0) / st.scale[0])
    assert st.amax_history[0, 0] == np.float32(np.abs(W).max())
    assert st.amax_cur[0] == np.float32(np.abs(W).max())


def test_quantize_weight_of_zeros_keeps_unit_scale():
    codes, sinv, st = omod.quantize_weight(np.zeros((16, 32), np.uint16), Recipe("hybrid", 4))
    assert not codes.any() and sinv == 1.0 and st.scale[0] == 1.0


def _ln_params(K, N, seed):
    return synth.linear_params(N, K, layer=seed, bias_std=0.02)


def test_linear_fp8_weight_branch_equals_bf16_branch():
    """Codes that the bf16 branch would cast (state scale[1]) give the same
    output and saved scale_inv; only slot 1's amax is left unrecorded."""
    M, K, N = 40, 64, 48
    p = _ln_params(K, N, 1)
    x = synth.activations(M, K, dist="outliers")
    rec = Recipe("hybrid", 4)
    st = ScalingState(2, 4)
    st.scale[:] = [3.5, 2000.0]
    st.scale_inv[:] = np.float32(1.0) / st.scale
    s1, s2 = st.copy(), st.copy()
    y1, c1, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], s1, rec, update=False)
    y2, c2, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], None, p["b"], s2, rec, update=False,
                                   fp8_weight=(c1.wq[0], st.scale_inv[1]))
    assert np.array_equal(y1, y2) and np.array_equal(c1.sinv, c2.sinv)
    assert s1.amax_cur[0] == s2.amax_cur[0] and s1.amax_cur[1] > 0 and s2.amax_cur[1] == 0


def test_mlp_fp8_weight_branch_equals_bf16_branch():
    M, D, F = 24, 32, 64
    p = synth.mlp_params(D, F, layer=2, bias_std=0.02)
    x = synth.activations(M, D, dist="outliers")
    rec = Recipe("hybrid", 4)
    st = ScalingState(4, 4)
    st.scale[:] = [4.0, 1500.0, 20.0, 900.0]  # distinct per slot: a slot mix-up changes the result
    st.scale_inv[:] = np.float32(1.0) / st.scale
    s1, s2 = st.copy(), st.copy()
    y1, c1, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], s1, rec, update=False)
    y2, c2, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], None, p["b1"], None, p["b2"], s2, rec, update=False,
                                fp8_weights=((c1.wq[0], st.scale_inv[1]), (c1.wq[1], st.scale_inv[3])))
    assert np.array_equal(y1, y2) and np.array_equal(c1.sinv, c2.sinv)
    assert np.array_equal(s1.amax_cur[[0, 2]], s2.amax_cur[[0, 2]])
    assert s2.amax_cur[1] == 0 and s2.amax_cur[3] == 0 and s1.amax_cur[1] > 0 and s1.amax_cur[3] > 0


def test_fp8_weight_forward_near_exact_layer():
    """With the weight's own scale (far from the state's unit scale), the output
    stays within FP8 quantisation error of the exact fp64 layer: a GEMM that took
    the state's scale_inv instead would be off by the weight's scale (~1e4)."""
    M, K, N = 64, 128, 96
    p = _ln_params(K, N, 3)
    x = synth.activations(M, K)
    rec = Recipe("hybrid", 4)
    codes, sinv, _ = omod.quantize_weight(p["w"], rec)
    assert sinv < 1e-3
    y, _, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], None, p["b"], ScalingState(2, 4), rec, update=False,
                                 fp8_weight=(codes, sinv))
    ye, _, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], ScalingState(2, 4), rec, exact=True,
                                  update=False)
    err = np.linalg.norm(y - ye) / np.linalg.norm(ye)
    assert err < 0.1, err


def test_exact_mode_refuses_fp8_weight():
    with pytest.raises(ValueError):
        omod.ln_linear_fwd(np.zeros((2, 16)), None, None, None, None, ScalingState(2, 1), Recipe(), exact=True,
                           fp8_weight=(np.zeros((16, 16), np.uint8), np.float32(1)))


# ---- the residual add ahead of a LayerNorm module
def _bf16_bits_sum_torch(a_bits, b_bits):
    """bf16 + bf16 -> bf16 by torch's own bf16 addition (an independent rounding)."""
    import torch
    ta = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b_bits.view(np.int16)).view(torch.bfloat16)
    return (ta + tb).view(torch.int16).numpy().view(np.uint16)


def test_residual_sum_matches_torch_bf16_addition_and_zero_is_identity():
    M, D, F = 24, 32, 64
    p = synth.mlp_params(D, F, layer=4, bias_std=0.02)
    x = synth.activations(M, D, dist="outliers", step=3)
    r = synth.activations(M, D, step=5, tid=synth.TID["attn"])
    rec = Recipe("hybrid", 4)
    h = _bf16_bits_sum_torch(x, r)
    y1, c1, a1 = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], ScalingState(4, 4), rec,
                                 update=False, residual=r)
    y2, c2, _ = omod.ln_mlp_fwd(h, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], ScalingState(4, 4), rec,
                                update=False)
    assert np.array_equal(a1["x_sum"], bf16_to_f32(h)) and np.array_equal(y1, y2) and np.array_equal(c1.x, c2.x)
    z = np.zeros_like(x)
    y3, _, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], ScalingState(4, 4), rec,
                               update=False, residual=z)
    y4, _, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], ScalingState(4, 4), rec,
                               update=False)
    assert np.array_equal(y3, y4)
    pl = synth.linear_params(48, D, layer=2, bias_std=0.02)
    ly1, _, la = omod.ln_linear_fwd(x, pl["gamma"], pl["beta"], pl["w"], pl["b"], ScalingState(2, 4), rec, update=False,
                                    residual=r)
    ly2, _, _ = omod.ln_linear_fwd(h, pl["gamma"], pl["beta"], pl["w"], pl["b"], ScalingState(2, 4), rec, update=False)
    assert np.array_equal(ly1, ly2) and np.array_equal(la["x_sum"], bf16_to_f32(h))
    with pytest.raises(ValueError):  # a residual needs the LayerNorm it precedes
        omod.ln_linear_fwd(x, None, None, pl["w"], pl["b"], ScalingState(2, 4), rec, residual=r)


def test_quantize_weight_hand_worked_cases():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fp8_weight_cases.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        fmt_name, margin, w, scale, codes, _ = [f.strip() for f in line.split("|", 5)]
        W = np.array([[float(v) for v in row.split()] for row in w.split(";")], dtype=np.float32)
        rec = Recipe(fmt_name if fmt_name != "e4m3" else "hybrid", 16, margin=int(margin))
        got, sinv, st = omod.quantize_weight(synth.f32_to_bf16_bits(W), rec)
        assert st.scale[0] == np.float32(float(scale)), line
        assert sinv == np.float32(np.float32(1.0) / np.float32(float(scale))), line
        assert [int(c, 16) for c in codes.split()] == got.ravel().tolist(), line
        n += 1
    assert n == 4
