"""FP8-stored weights (fp8_model_init, TE tutorial closing list) on the GPU.

The one-time conversion is an integer decision taken in fp32 on both sides, so
codes, scale_inv and the weight's state must match the oracle bit for bit. The
forward then runs with no weight cast: its output is compared with the oracle
fed the same codes (1e-2 relative Frobenius), its state after the update with
the oracle state machine fed the amaxes the GPU recorded (bit for bit; the
weight slots record nothing), and its launch count is one cast fewer. A
backward after such a forward uses the weight's own scale_inv.
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import modules as omod
from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
from helpers import bf16_dev, host, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _state(meta):
    s = ScalingState(meta.n, meta.history_len)
    s.scale[:] = host(meta.scale)
    s.scale_inv[:] = host(meta.scale_inv)
    s.amax_history[:] = host(meta.amax_history)
    s.amax_cur[:] = host(meta.amax_cur)
    return s


def _bits_equal(meta, st):
    for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
        g = host(getattr(meta, name)).astype(np.float32)
        if not np.array_equal(g.view(np.uint32), getattr(st, name).view(np.uint32)):
            return False
    return True


@pytest.mark.parametrize("rows,cols", [(2304, 768), (768, 3072), (208, 48), (0, 64)])
@pytest.mark.parametrize("fmt,margin", [("hybrid", 0), ("e5m2", 0), ("hybrid", 2)])
def test_quantize_weight_bit_exact(L, rows, cols, fmt, margin):
    w = synth.linear_params(rows, cols, ln=False, layer=rows % 7)["w"]
    rec, orec = L.Recipe(fmt, 16, margin=margin), ORecipe(fmt, 16, margin=margin)
    fw = L.quantize_weight(bf16_dev(w), rec)
    L.sync_status()
    codes, sinv, st = omod.quantize_weight(w, orec, ScalingState(1, 1))
    assert np.array_equal(host(fw.codes), codes)
    assert host(fw.scale_inv).astype(np.float32).view(np.uint32)[0] == np.float32(sinv).view(np.uint32)
    assert _bits_equal(fw.meta, st)


@pytest.mark.parametrize("M,ln", [(512, True), (1000, True), (264, False)])
def test_linear_fwd_with_fp8_weight(L, M, ln):
    K, N = 768, 2304
    rec, orec = L.Recipe("hybrid", 16), ORecipe("hybrid", 16)
    ff = orec.fwd_fmt()
    p = synth.linear_params(N, K, ln=ln, layer=1, bias_std=0.02)
    fw = L.quantize_weight(bf16_dev(p["w"]), rec)
    codes0 = fw.codes.clone()
    wcodes, wsinv, _ = omod.quantize_weight(p["w"], orec)  # the oracle's own conversion
    assert np.array_equal(host(fw.codes), wcodes)
    meta = L.ScalingMeta(2, 16)
    gmeta = L.ScalingMeta(1, 16)
    g = bf16_dev(p["gamma"]) if ln else None
    be = bf16_dev(p["beta"]) if ln else None
    for step in range(3):
        x = synth.activations(M, K, dist="outliers", step=step)
        pre = _state(meta)
        n0 = L.launch_count()
        y, ctx = L.ln_linear_fwd(bf16_dev(x), g, be, fw, bf16_dev(p["b"]), meta, rec, defer_update=True)
        assert L.launch_count() - n0 == 2  # LayerNorm (or input) cast, GEMM: no weight cast
        oy, octx, _ = omod.ln_linear_fwd(x, p["gamma"] if ln else None, p["beta"] if ln else None, None, p["b"],
                                         pre.copy(), orec, update=False, fp8_weight=(wcodes, wsinv))
        assert rel_fro(host(y), oy) < TOL, step
        got = _state(meta)
        assert got.amax_cur[1] == pre.amax_cur[1] == 0  # no weight amax recorded
        sinv_saved = host(ctx.sinv_saved).astype(np.float32)
        assert sinv_saved[1] == wsinv and sinv_saved[0] == pre.scale_inv[0]
        # the backward after an FP8-weight forward dequantises dgrad with the weight's own scale_inv
        dy = synth.grad(M, N, step=step)
        gpre = _state(gmeta)
        gr = L.ln_linear_bwd(bf16_dev(dy), bf16_dev(x), g, ctx, gmeta, rec)
        og = omod.ln_linear_bwd(dy, octx, gpre.copy(), orec, update=False)
        for k in ("dx", "dw") + (("dgamma",) if ln else ()):
            assert rel_fro(host(getattr(gr, k)), og[k]) < TOL, (step, k)
        L.amax_history_update(meta, rec, [L.E4M3, L.E4M3])
        L.sync_status()
        tf = pre.copy()
        tf.record(0, got.amax_cur[0])
        tf.update([ff, ff])
        assert _bits_equal(meta, tf), step
        assert torch.equal(fw.codes, codes0)  # the stored codes are read only


@pytest.mark.parametrize("M,fused", [(512, False), (1000, False), (512, True), (8192, True)])
def test_mlp_fwd_with_fp8_weights(L, M, fused):
    D, F = 768, 3072
    rec, orec = L.Recipe("hybrid", 16), ORecipe("hybrid", 16)
    ff = orec.fwd_fmt()
    p = synth.mlp_params(D, F, layer=3, bias_std=0.02)
    f1, f2 = L.quantize_weight(bf16_dev(p["w1"]), rec), L.quantize_weight(bf16_dev(p["w2"]), rec)
    ow = (omod.quantize_weight(p["w1"], orec)[:2], omod.quantize_weight(p["w2"], orec)[:2])
    assert np.array_equal(host(f1.codes), ow[0][0]) and np.array_equal(host(f2.codes), ow[1][0])
    meta = L.ScalingMeta(4, 16)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    for step in range(2):
        x = synth.activations(M, D, dist="outliers", step=step)
        pre = _state(meta)
        ctx = L.mlp_ctx(M, D, F, fused=fused, weight_codes=False)
        n0 = L.launch_count()
        y, ctx = L.ln_mlp_fwd(bf16_dev(x), dev["gamma"], dev["beta"], f1, dev["b1"], f2, dev["b2"], meta, rec,
                              ctx=ctx, defer_update=True)
        # LayerNorm cast and two GEMMs; when fused, one launch for both GEMMs and the LayerNorm
        # launch clears their readiness counters
        assert L.launch_count() - n0 == (2 if fused else 3)
        oy, _, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], None, p["b1"], None, p["b2"], pre.copy(), orec,
                                   update=False, fp8_weights=ow)
        assert rel_fro(host(y), oy) < TOL, step
        got = _state(meta)
        assert got.amax_cur[1] == 0 and got.amax_cur[3] == 0
        ss = host(ctx.sinv_saved).astype(np.float32)
        assert ss[1] == ow[0][1] and ss[3] == ow[1][1] and ss[0] == pre.scale_inv[0] and ss[2] == pre.scale_inv[2]
        L.amax_history_update(meta, rec, [L.E4M3] * 4)
        L.sync_status()
        tf = pre.copy()
        tf.record(0, got.amax_cur[0])
        tf.record(2, got.amax_cur[2])
        tf.update([ff] * 4)
        assert _bits_equal(meta, tf), step


def test_fp8_weight_argument_errors(L):
    rec = L.Recipe("hybrid", 16)
    f1 = L.quantize_weight(bf16_dev(synth.linear_params(64, 32, ln=False)["w"]), rec)
    p = synth.mlp_params(32, 64)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    with pytest.raises(TypeError):
        L.ln_mlp_fwd(bf16_dev(synth.activations(16, 32)), dev["gamma"], dev["beta"], f1, None, dev["w2"], None,
                     L.ScalingMeta(4, 16), rec)
    with pytest.raises(L.LnFp8Error):
        L.quantize_weight(bf16_dev(synth.linear_params(64, 32, ln=False)["w"]), rec, meta=L.ScalingMeta(2, 16))
