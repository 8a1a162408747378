"""The residual add fused ahead of the LayerNorm of LayerNormLinear and
LayerNormMLP (GPU).

The module input h = bf16(x + r) is a rounding decision both sides take from
the same two bf16 tensors, so the x_sum the kernel writes must equal the
oracle's sum bit for bit; the module outputs and, with x_sum as the backward's
x, the gradients are compared with the oracle module fed x and r (1e-2 relative
Frobenius); and the fused call equals, bit for bit, the plain call fed x_sum.
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import modules as omod
from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
from oracle.gemm import to_bf16_bits
from helpers import bf16_dev, host, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,D,F", [(512, 768, 3072), (1000, 768, 3072), (264, 2048, 8192)])
def test_mlp_forward_backward_with_fused_residual(L, M, D, F):
    rec, orec = L.Recipe("hybrid", 16), ORecipe("hybrid", 16)
    p = synth.mlp_params(D, F, layer=5, bias_std=0.02)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    x = synth.activations(M, D, dist="outliers", step=1)
    r = synth.activations(M, D, step=2, tid=synth.TID["attn"])
    dy = synth.grad(M, D, step=1)
    fm, bm = L.ScalingMeta(4, 16), L.ScalingMeta(2, 16)
    y, ctx = L.ln_mlp_fwd(bf16_dev(x), dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm, rec,
                          residual=bf16_dev(r))
    g = L.ln_mlp_bwd(bf16_dev(dy), ctx.x_sum, dev["gamma"], ctx, bm, rec)
    L.sync_status()
    oy, octx, aux = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], ScalingState(4, 16),
                                    orec, residual=r)
    og = omod.ln_mlp_bwd(dy, octx, ScalingState(2, 16), orec)
    assert np.array_equal(_bits(ctx.x_sum), to_bf16_bits(aux["x_sum"]))
    assert rel_fro(host(y), oy) < TOL
    for k in ("dx", "dw1", "dw2", "dgamma"):
        assert rel_fro(host(getattr(g, k)), og[k]) < TOL, k
    # the plain call fed x_sum runs the same arithmetic
    fm2 = L.ScalingMeta(4, 16)
    y2, ctx2 = L.ln_mlp_fwd(ctx.x_sum.clone(), dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm2,
                            rec)
    L.sync_status()
    assert torch.equal(y2, y) and torch.equal(ctx2.lnq, ctx.lnq) and torch.equal(fm2.amax_history, fm.amax_history)


@pytest.mark.parametrize("M", [264, 1000])
def test_linear_forward_with_fused_residual(L, M):
    K, N = 768, 2304
    rec, orec = L.Recipe("hybrid", 16), ORecipe("hybrid", 16)
    p = synth.linear_params(N, K, layer=6, bias_std=0.02, wtid=synth.TID["wqkv"], btid=synth.TID["bqkv"])
    x = synth.activations(M, K, dist="outliers", step=4)
    r = synth.activations(M, K, step=3, tid=synth.TID["attn"])
    dy = synth.grad(M, N, step=4)
    fm, bm = L.ScalingMeta(2, 16), L.ScalingMeta(1, 16)
    g_, b_ = bf16_dev(p["gamma"]), bf16_dev(p["beta"])
    y, ctx = L.ln_linear_fwd(bf16_dev(x), g_, b_, bf16_dev(p["w"]), bf16_dev(p["b"]), fm, rec, residual=bf16_dev(r))
    gr = L.ln_linear_bwd(bf16_dev(dy), ctx.x_sum, g_, ctx, bm, rec)
    L.sync_status()
    oy, octx, aux = omod.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], ScalingState(2, 16), orec, residual=r)
    og = omod.ln_linear_bwd(dy, octx, ScalingState(1, 16), orec)
    assert np.array_equal(_bits(ctx.x_sum), to_bf16_bits(aux["x_sum"]))
    assert rel_fro(host(y), oy) < TOL
    for k in ("dx", "dw", "dgamma"):
        assert rel_fro(host(getattr(gr, k)), og[k]) < TOL, k


def test_residual_without_layernorm_is_refused(L):
    rec = L.Recipe("hybrid", 16)
    p = synth.linear_params(64, 32, ln=False)
    x = bf16_dev(synth.activations(16, 32))
    with pytest.raises(L.LnFp8Error):
        L.ln_linear_fwd(x, None, None, bf16_dev(p["w"]), None, L.ScalingMeta(2, 16), rec, residual=x)
