"""A stack of transformer-block FP8 modules, several steps (GPU).

Each of the stack's layers runs the block the pages' model is built from,
around a synthetic attention output (attention itself is not on the path):

    qkv = LayerNormLinear(h)            768 -> 2304 (discarded: attention is synthetic)
    h   = h + Linear(attn)              768 -> 768 on attn ~ N(0, 1)
    h   = h + LayerNormMLP(h)           768 -> 3072 -> 768

and the backward in reverse with synthetic dQKV ~ N(0, 0.01) and the residual
gradient flowing through. On the GPU side the residual adds in front of the
MLP's and the next layer's LayerNorm run fused into those LayerNorm kernels
(their x_sum must equal the oracle's residual stream bit for bit). Every module call defers its state update; after the
step one ``amax_history_update_many`` launch updates all layers' forward and
backward states. The oracle runs the whole stack on its own (its own residual
stream and its own state machines); the GPU modules take the oracle stream's
values as inputs, so no oracle input comes from the GPU. The checks, per step
and layer: every module output and gradient against the oracle module (1e-2
relative Frobenius); the recorded amaxes and the states after the one-launch
update against the oracle's own, bit for bit where both sides reduce the same
bf16 values (weights, Linear inputs, dY) and within a stated relative bound
where the amax is of an fp32 intermediate; and the update kernel alone, bit for
bit, against the oracle rule applied to the GPU's pre-update state. The residual
adds round to bf16 in numpy.
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import modules as omod
from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
from oracle.gemm import bf16_to_f32, to_bf16_bits
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


def _bf16_add(a, b):
    """bf16(a + b) of two bf16-valued float arrays (the residual add)."""
    return bf16_to_f32(to_bf16_bits(np.asarray(a, np.float64) + np.asarray(b, np.float64))).astype(np.float64)


def _to_bits(v):
    return to_bf16_bits(np.asarray(v, np.float64))


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _close_state(meta, st, rtol):
    """GPU state against the oracle's own within rtol (amaxes of fp32 intermediates)."""
    for name in ("scale", "scale_inv", "amax_history"):
        g = host(getattr(meta, name)).astype(np.float64)
        o = getattr(st, name).astype(np.float64)
        if not np.allclose(g, o, rtol=rtol, atol=0):
            return False
    return True


# Slots whose amax is max|t| of a tensor both sides hold bit for bit (weights, the bf16 inputs
# of Linear and of every backward) are compared bit for bit; the others (LayerNorm output, GELU
# output, dH: fp32 values computed in a different order) within a relative tolerance.
EXACT = {"fq": [False, True], "fp": [True, True], "fm": [False, True, False, True], "bq": [True], "bp": [True],
         "bm": [True, False]}
RTOL = {"fq": 1e-5, "fp": 0.0, "fm": 1e-2, "bq": 0.0, "bp": 0.0, "bm": 1e-2}


@pytest.mark.parametrize("layers,M,steps", [(4, 512, 3)])
def test_block_stack_with_one_state_update_launch(L, layers, M, steps):
    D, F, NQKV = 768, 3072, 2304
    rec, orec = L.Recipe("hybrid", 16), ORecipe("hybrid", 16)
    ff, gf = orec.fwd_fmt(), orec.bwd_fmt()
    E4, E5 = L.E4M3, L.E5M2
    P = []
    for l in range(layers):
        P.append(dict(
            qkv=synth.linear_params(NQKV, D, layer=l, bias_std=0.02, wtid=synth.TID["wqkv"], btid=synth.TID["bqkv"]),
            proj=synth.linear_params(D, D, layer=l, ln=False, bias_std=0.02, wtid=synth.TID["wproj"],
                                     btid=synth.TID["bproj"]),
            mlp=synth.mlp_params(D, F, layer=l, bias_std=0.02)))
    dev = [dict(qkv={k: (bf16_dev(v) if v is not None else None) for k, v in p["qkv"].items()},
                proj={k: (bf16_dev(v) if v is not None else None) for k, v in p["proj"].items()},
                mlp={k: bf16_dev(v) for k, v in p["mlp"].items()}) for p in P]
    # per layer: forward metas (qkv 2, proj 2, mlp 4) and backward metas (1, 1, 2)
    M_ = [dict(fq=L.ScalingMeta(2, 16), fp=L.ScalingMeta(2, 16), fm=L.ScalingMeta(4, 16),
               bq=L.ScalingMeta(1, 16), bp=L.ScalingMeta(1, 16), bm=L.ScalingMeta(2, 16)) for _ in range(layers)]
    order = ["fq", "fp", "fm", "bq", "bp", "bm"]
    # the oracle's own states, run next to the GPU's from the same initial state
    O_ = [{k: ScalingState(m[k].n, 16) for k in order} for m in M_]
    dts = {"fq": [E4, E4], "fp": [E4, E4], "fm": [E4] * 4, "bq": [E5], "bp": [E5], "bm": [E5, E5]}
    ofmts = {"fq": [ff] * 2, "fp": [ff] * 2, "fm": [ff] * 4, "bq": [gf], "bp": [gf], "bm": [gf] * 2}
    for step in range(steps):
        # the residual stream is the oracle's: both sides get its values at every layer
        h = bf16_to_f32(synth.activations(M, D, dist="outliers", step=step)).astype(np.float64)
        saved = []
        prev = None  # (residual stream before the last MLP add, that MLP's output) as bf16 bits
        for l in range(layers):
            p, d, m, o = P[l], dev[l], M_[l], O_[l]
            hb = _to_bits(h)
            attn = synth.activations(M, D, step=step, tid=synth.TID["attn"], layer=l)
            if prev is None:
                xq = bf16_dev(hb)
                qkv, cq = L.ln_linear_fwd(xq, d["qkv"]["gamma"], d["qkv"]["beta"], d["qkv"]["w"], d["qkv"]["b"],
                                          m["fq"], rec, defer_update=True)
            else:  # the previous MLP's residual add fused into this LayerNorm
                qkv, cq = L.ln_linear_fwd(bf16_dev(prev[0]), d["qkv"]["gamma"], d["qkv"]["beta"], d["qkv"]["w"],
                                          d["qkv"]["b"], m["fq"], rec, defer_update=True, residual=bf16_dev(prev[1]))
                assert np.array_equal(_bits(cq.x_sum), hb), (step, l, "qkv residual")
                xq = cq.x_sum
            oq_y, ocq, _ = omod.ln_linear_fwd(hb, p["qkv"]["gamma"], p["qkv"]["beta"], p["qkv"]["w"], p["qkv"]["b"],
                                              o["fq"], orec, update=False)
            assert rel_fro(host(qkv), oq_y) < TOL, (step, l, "qkv")
            xa = bf16_dev(attn)
            pr, cp = L.ln_linear_fwd(xa, None, None, d["proj"]["w"], d["proj"]["b"], m["fp"], rec, defer_update=True)
            op_y, ocp, _ = omod.ln_linear_fwd(attn, None, None, p["proj"]["w"], p["proj"]["b"], o["fp"], orec,
                                              update=False)
            assert rel_fro(host(pr), op_y) < TOL, (step, l, "proj")
            h = _bf16_add(h, op_y)
            hb2 = _to_bits(h)
            # the projection's residual add fused into the MLP's LayerNorm
            y, cm = L.ln_mlp_fwd(bf16_dev(hb), d["mlp"]["gamma"], d["mlp"]["beta"], d["mlp"]["w1"], d["mlp"]["b1"],
                                 d["mlp"]["w2"], d["mlp"]["b2"], m["fm"], rec, defer_update=True,
                                 residual=bf16_dev(_to_bits(op_y)))
            assert np.array_equal(_bits(cm.x_sum), hb2), (step, l, "mlp residual")
            xm = cm.x_sum
            om_y, ocm, _ = omod.ln_mlp_fwd(hb2, p["mlp"]["gamma"], p["mlp"]["beta"], p["mlp"]["w1"], p["mlp"]["b1"],
                                           p["mlp"]["w2"], p["mlp"]["b2"], o["fm"], orec, update=False)
            assert rel_fro(host(y), om_y) < TOL, (step, l, "mlp")
            h = _bf16_add(h, om_y)
            prev = (hb2, _to_bits(om_y))
            saved.append((xq, cq, ocq, xa, cp, ocp, xm, cm, ocm))
        dh = bf16_to_f32(synth.grad(M, D, step=step)).astype(np.float64)
        for l in reversed(range(layers)):
            p, d, m, o = P[l], dev[l], M_[l], O_[l]
            xq, cq, ocq, xa, cp, ocp, xm, cm, ocm = saved[l]
            g = L.ln_mlp_bwd(bf16_dev(_to_bits(dh)), xm, d["mlp"]["gamma"], cm, m["bm"], rec, defer_update=True)
            og = omod.ln_mlp_bwd(_to_bits(dh), ocm, o["bm"], orec, update=False)
            for k in ("dx", "dw1", "dw2", "dgamma"):
                assert rel_fro(host(getattr(g, k)), og[k]) < TOL, (step, l, "mlp", k)
            dh = _bf16_add(dh, og["dx"])
            gp = L.ln_linear_bwd(bf16_dev(_to_bits(dh)), xa, None, cp, m["bp"], rec, defer_update=True)
            ogp = omod.ln_linear_bwd(_to_bits(dh), ocp, o["bp"], orec, update=False)
            assert rel_fro(host(gp.dw), ogp["dw"]) < TOL, (step, l, "proj dw")
            dqkv = synth.grad(M, NQKV, step=step, layer=l, tid=synth.TID["attn"])
            gq = L.ln_linear_bwd(bf16_dev(dqkv), xq, d["qkv"]["gamma"], cq, m["bq"], rec, defer_update=True)
            ogq = omod.ln_linear_bwd(dqkv, ocq, o["bq"], orec, update=False)
            for k in ("dx", "dw", "dgamma"):
                assert rel_fro(host(getattr(gq, k)), ogq[k]) < TOL, (step, l, "qkv", k)
            dh = _bf16_add(dh, ogq["dx"])
        L.sync_status()
        # the recorded amaxes: bit for bit where both sides reduce the same values
        for l in range(layers):
            for k in order:
                ga = host(M_[l][k].amax_cur).astype(np.float32)
                oa = O_[l][k].amax_cur
                for i in range(len(ga)):
                    if EXACT[k][i]:
                        assert ga[i].view(np.uint32) == oa[i].view(np.uint32), (step, l, k, i)
                    else:
                        assert abs(float(ga[i]) - float(oa[i])) <= RTOL[k] * float(oa[i]), (step, l, k, i)
        # one launch for every layer's six states
        pre = [{k: _state(m[k]) for k in order} for m in M_]
        metas = [m[k] for m in M_ for k in order]
        L.amax_history_update_many(metas, rec, [dts[k] for _ in M_ for k in order])
        L.sync_status()
        for l in range(layers):
            for k in order:
                O_[l][k].update(ofmts[k])
                # against the oracle's own state machine
                if all(EXACT[k]):
                    assert _bits_equal(M_[l][k], O_[l][k]), (step, l, k)
                else:
                    assert _close_state(M_[l][k], O_[l][k], RTOL[k]), (step, l, k)
                # the update kernel on its own: the GPU's pre-update state through the oracle rule
                tf = pre[l][k].copy()
                tf.update(ofmts[k])
                assert _bits_equal(M_[l][k], tf), (step, l, k, "update rule")


@pytest.mark.parametrize("ns,hist", [((1, 2, 4, 3), 8), (tuple(1 + k % 4 for k in range(128)), 1024)])
def test_update_many_equals_separate_updates(L, ns, hist):
    rec = L.Recipe("hybrid", hist)
    rng = np.random.default_rng(3)
    metas = [L.ScalingMeta(n, hist) for n in ns]
    twins = [L.ScalingMeta(m.n, hist) for m in metas]
    dts = [[L.E4M3] * m.n if i % 2 == 0 else [L.E5M2] * m.n for i, m in enumerate(metas)]
    for step in range(5):
        for m, t in zip(metas, twins):
            a = torch.tensor((rng.random(m.n) * 10.0 ** rng.integers(-3, 3)).astype(np.float32), device="cuda")
            m.amax_cur.copy_(a)
            t.amax_cur.copy_(a)
        snaps = [torch.zeros(m.n, device="cuda") for m in metas]
        before = [m.scale_inv.clone() for m in metas]
        L.amax_history_update_many(metas, rec, dts, scale_inv_before=snaps)
        for t, d in zip(twins, dts):
            L.amax_history_update(t, rec, d)
        L.sync_status()
        for m, t in zip(metas, twins):
            for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
                assert torch.equal(getattr(m, name), getattr(t, name)), (step, name)
        for sn, b in zip(snaps, before):
            assert torch.equal(sn, b), step
    L.amax_history_update_many([], rec, [])  # nothing to do
    with pytest.raises(L.LnFp8Error):  # more sets than one launch takes
        L.amax_history_update_many(metas + metas[:1] * (129 - len(metas)), rec, dts + dts[:1] * (129 - len(metas)))
    with pytest.raises(L.LnFp8Error):  # a set listed twice would race with itself
        L.amax_history_update_many([metas[0], metas[1], metas[0]], rec, [dts[0], dts[1], dts[0]])
