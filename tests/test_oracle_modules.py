"""Pins of the oracle's LayerNormLinear / Linear / LayerNormMLP composition (CPU).

With quantisation and intermediate roundings switched off (``exact=True``) the
modules must reduce to the textbook fp64 LayerNorm -> Linear (-> GELU -> Linear)
and its autograd gradients (TE tutorial, code block 2: the plain-PyTorch block
``nn.LayerNorm`` + ``nn.Sequential(nn.Linear, nn.GELU(), nn.Linear)``). A
transposed operand, a wrong scale pairing or a dropped term in the dataflow
fails these. With quantisation on, the results are checked for the properties
that hold by construction (amaxes recorded, codes equal the cast of the
recorded pre-cast values, error of the order of the FP8 precision).
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8, modules
from oracle.delayed_scaling import Recipe, ScalingState

torch = pytest.importorskip("torch")


def _mlp_inputs(m, d, f, seed=3):
    p = synth.mlp_params(d, f, seed=seed, bias_std=0.05)
    x = synth.activations(m, d, dist="outliers", seed=seed)
    dy = synth.grad(m, d, seed=seed)
    return x, dy, p


def _t(bits):
    return torch.from_numpy(synth.bf16_bits_to_f32(bits).astype(np.float64))


@pytest.mark.parametrize("approx", ["tanh", "erf"])
def test_exact_mlp_equals_fp64_autograd(approx):
    m, d, f = 24, 16, 40
    x, dy, p = _mlp_inputs(m, d, f)
    rec = Recipe()
    Y, ctx, _ = modules.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"],
                                   ScalingState(4, 16), rec, exact=True, gelu_approx=approx)
    g = modules.ln_mlp_bwd(dy, ctx, ScalingState(2, 16), rec, exact=True, gelu_approx=approx)

    X = _t(x).requires_grad_()
    G, B = _t(p["gamma"]).requires_grad_(), _t(p["beta"]).requires_grad_()
    W1, B1 = _t(p["w1"]).requires_grad_(), _t(p["b1"]).requires_grad_()
    W2, B2 = _t(p["w2"]).requires_grad_(), _t(p["b2"]).requires_grad_()
    h = torch.nn.functional.layer_norm(X, (d,), G, B, eps=1e-5) @ W1.T + B1
    a = torch.nn.functional.gelu(h, approximate="tanh" if approx == "tanh" else "none")
    y = a @ W2.T + B2
    y.backward(_t(dy))
    tol = dict(rtol=1e-9, atol=1e-12)
    assert np.allclose(Y, y.detach().numpy(), **tol)
    for name, ref in [("dx", X), ("dgamma", G), ("dbeta", B), ("dw1", W1), ("db1", B1), ("dw2", W2), ("db2", B2)]:
        assert np.allclose(g[name], ref.grad.numpy(), **tol), name


@pytest.mark.parametrize("with_ln", [True, False])
def test_exact_linear_equals_fp64_autograd(with_ln):
    m, k, n = 20, 24, 36
    p = synth.linear_params(n, k, ln=with_ln, bias_std=0.05, seed=4)
    x = synth.activations(m, k, seed=4)
    dy = synth.grad(m, n, seed=4)
    rec = Recipe()
    Y, ctx, _ = modules.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], ScalingState(2, 16), rec, exact=True)
    g = modules.ln_linear_bwd(dy, ctx, ScalingState(1, 16), rec, exact=True)
    X = _t(x).requires_grad_()
    W, Bb = _t(p["w"]).requires_grad_(), _t(p["b"]).requires_grad_()
    if with_ln:
        G, B = _t(p["gamma"]).requires_grad_(), _t(p["beta"]).requires_grad_()
        u = torch.nn.functional.layer_norm(X, (k,), G, B, eps=1e-5)
    else:
        u = X
    y = u @ W.T + Bb
    y.backward(_t(dy))
    tol = dict(rtol=1e-9, atol=1e-12)
    assert np.allclose(Y, y.detach().numpy(), **tol)
    assert np.allclose(g["dx"], X.grad.numpy(), **tol)
    assert np.allclose(g["dw"], W.grad.numpy(), **tol)
    assert np.allclose(g["db"], Bb.grad.numpy(), **tol)
    if with_ln:
        assert np.allclose(g["dgamma"], G.grad.numpy(), **tol)
        assert np.allclose(g["dbeta"], B.grad.numpy(), **tol)


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def test_quantised_mlp_records_amaxes_and_casts_what_it_recorded():
    m, d, f = 64, 32, 96
    x, dy, p = _mlp_inputs(m, d, f, seed=8)
    rec = Recipe(amax_history_len=4)
    fs, bs = ScalingState(4, 4), ScalingState(2, 4)
    for step in range(3):
        xs = synth.activations(m, d, dist="outliers", seed=8, step=step)
        dys = synth.grad(m, d, seed=8, step=step)
        scale_before = fs.scale.copy()
        gscale_before = bs.scale.copy()
        Y, ctx, aux = modules.ln_mlp_fwd(xs, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs, rec)
        g = modules.ln_mlp_bwd(dys, ctx, bs, rec)
        # the history's newest row holds this step's amaxes
        assert fs.amax_history[0, 0] == fp8.amax(aux["y"])
        assert fs.amax_history[0, 2] == fp8.amax(aux["a"])
        assert fs.amax_history[0, 1] == fp8.amax(synth.bf16_bits_to_f32(p["w1"]))
        assert bs.amax_history[0, 0] == fp8.amax(synth.bf16_bits_to_f32(dys))
        assert bs.amax_history[0, 1] == fp8.amax(g["dh"])
        # the codes are the casts, with the scale in force before the update, of the recorded values
        assert np.array_equal(ctx.yq, fp8.quantize(aux["y"], scale_before[0], fp8.E4M3))
        assert np.array_equal(ctx.aq, fp8.quantize(aux["a"], scale_before[2], fp8.E4M3))
        assert np.array_equal(g["dhq"], fp8.quantize(g["dh"], gscale_before[1], fp8.E5M2))
        assert np.array_equal(ctx.sinv, 1 / scale_before.astype(np.float32)) or step == 0
        # quantised results stay within FP8 precision of the exact ones
        Ye, ctxe, _ = modules.ln_mlp_fwd(xs, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"],
                                         ScalingState(4, 4), rec, exact=True)
        ge = modules.ln_mlp_bwd(dys, ctxe, ScalingState(2, 4), rec, exact=True)
        assert _rel(Y, Ye) < 0.08
        if step > 0:  # after step 1 the scales use the dynamic range; step 1 casts at scale 1
            for k in ("dx", "dw1", "dw2", "db1"):
                assert _rel(g[k], ge[k]) < 0.15, k
