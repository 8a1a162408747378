"""LayerNormMLP / LayerNormLinear / Linear forward + backward through the C ABI
against the CPU oracle, over several delayed-scaling steps (GPU).

Each step is checked three ways:
  * step by step on the GPU's own intermediates (codes bit-exact against the
    oracle's cast of the kernel's fp32 pre-cast dumps, GEMMs against the
    oracle's GEMM of the GPU's codes);
  * end to end against an independent oracle run from the same inputs and the
    same (teacher-forced) pre-step state: bf16 outputs and gradients within
    1e-2 relative Frobenius error;
  * the delayed-scaling state after the step equals, bit for bit, the oracle's
    state machine fed the amaxes the GPU recorded; amaxes of exact inputs (the
    weights, dY) equal the oracle's bit for bit, amaxes of computed tensors
    agree within 2e-3 (LN output) and 1e-2 (GELU output, dH).
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8 as ofp8
from oracle import gelu as ogelu
from oracle import modules as omod
from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
from oracle.gemm import bf16_to_f32, dequant_scale, to_bf16_bits
from helpers import bf16_dev, host, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _state_from_gpu(meta):
    s = ScalingState(meta.n, meta.history_len)
    s.scale[:] = host(meta.scale)
    s.scale_inv[:] = host(meta.scale_inv)
    s.amax_history[:] = host(meta.amax_history)
    s.amax_cur[:] = host(meta.amax_cur)
    return s


def _assert_state_equal(meta, ost, what):
    for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
        g = host(getattr(meta, name)).astype(np.float32)
        assert np.array_equal(g.view(np.uint32), getattr(ost, name).view(np.uint32)), (what, name)


def _teacher_forced(pre: ScalingState, meta, fmts):
    """The oracle state machine run from the pre-step state with the amaxes the GPU recorded."""
    st = pre.copy()
    am = host(meta.amax_history)[0].astype(np.float32)
    for i in range(st.n):
        st.record(i, am[i])
    st.update(fmts)
    return st


def _bf16(x):
    return bf16_to_f32(to_bf16_bits(x)).astype(np.float64)


def _rel_amax(a, b):
    return abs(float(a) - float(b)) / max(abs(float(b)), 1e-30)


def run_mlp(L, M, D, F, steps, fmt="hybrid", hist=4, dist="outliers", bias_std=0.02, seed=11, full_check_steps=None,
            sample_rows=None):
    rec = L.Recipe(fmt, hist)
    orec = ORecipe(fmt, hist)
    p = synth.mlp_params(D, F, seed=seed, bias_std=bias_std)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    fm, bm = L.ScalingMeta(4, hist), L.ScalingMeta(2, hist)
    ffmt, gfmt = orec.fwd_fmt(), orec.bwd_fmt()
    full_check_steps = range(steps) if full_check_steps is None else full_check_steps
    ctx = L.mlp_ctx(M, D, F, debug=True)
    grads = L.mlp_grads(M, D, F, debug=True)
    for step in range(steps):
        x = synth.activations(M, D, dist=dist, seed=seed, step=step)
        dy = synth.grad(M, D, seed=seed, step=step)
        xt, dyt = bf16_dev(x), bf16_dev(dy)
        fpre, bpre = _state_from_gpu(fm), _state_from_gpu(bm)
        y, _ = L.ln_mlp_fwd(xt, dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm, rec, ctx=ctx)
        g = L.ln_mlp_bwd(dyt, xt, dev["gamma"], ctx, bm, rec, grads=grads)
        L.sync_status()

        # state: bit-exact against the oracle state machine fed the GPU's amaxes
        _assert_state_equal(fm, _teacher_forced(fpre, fm, [ffmt] * 4), f"fwd step {step}")
        _assert_state_equal(bm, _teacher_forced(bpre, bm, [gfmt] * 2), f"bwd step {step}")
        am_f = host(fm.amax_history)[0]
        am_b = host(bm.amax_history)[0]
        W1, W2 = bf16_to_f32(p["w1"]), bf16_to_f32(p["w2"])
        assert am_f[1] == ofp8.amax(W1) and am_f[3] == ofp8.amax(W2)
        assert am_b[0] == ofp8.amax(bf16_to_f32(dy))
        sc, gsc = fpre.scale, bpre.scale
        si, gsi = fpre.scale_inv, bpre.scale_inv
        assert np.array_equal(host(ctx.sinv_saved).view(np.uint32), si.view(np.uint32))

        # weights: exact inputs -> bit-exact codes
        assert np.array_equal(host(ctx.w1q), ofp8.quantize(W1, sc[1], ffmt))
        assert np.array_equal(host(ctx.w2q), ofp8.quantize(W2, sc[3], ffmt))

        if step not in full_check_steps:
            continue
        rows = np.arange(M) if sample_rows is None else sample_rows
        # ---- step-by-step on the GPU's intermediates
        ydbg = host(ctx.ln_out_debug)
        lnq = host(ctx.lnq)
        assert np.array_equal(lnq, ofp8.quantize(ydbg, sc[0], ffmt))
        assert am_f[0] == ofp8.amax(ydbg)
        hq = host(ctx.h)
        w1q, w2q = host(ctx.w1q), host(ctx.w2q)
        h_ref = ofp8.decode(lnq[rows], ffmt) @ ofp8.decode(w1q, ffmt).T * np.float64(dequant_scale(si[0], si[1])) \
            + bf16_to_f32(p["b1"])[None, :]
        assert np.abs(hq[rows] - h_ref).max() <= 2.0 ** -7 * np.abs(h_ref).max() + 1e-6
        assert rel_fro(hq[rows], _bf16(h_ref)) < 1e-3
        adbg = host(ctx.act_debug)
        a_ref = ogelu.gelu(hq[rows])
        assert np.abs(adbg[rows] - a_ref).max() <= 2e-3 * np.abs(a_ref).max()
        aq = host(ctx.aq)
        assert np.array_equal(aq, ofp8.quantize(adbg, sc[2], ffmt))
        assert am_f[2] == ofp8.amax(adbg)
        yv = host(y)
        y_ref = ofp8.decode(aq[rows], ffmt) @ ofp8.decode(w2q, ffmt).T * np.float64(dequant_scale(si[2], si[3])) \
            + bf16_to_f32(p["b2"])[None, :]
        assert rel_fro(yv[rows], _bf16(y_ref)) < 1e-3
        dyq = host(g.dyq)
        assert np.array_equal(dyq, ofp8.quantize(bf16_to_f32(dy), gsc[0], gfmt))
        dhd = host(g.dh_debug)
        da_ref = ofp8.decode(dyq[rows], gfmt) @ ofp8.decode(w2q, ffmt) * np.float64(dequant_scale(gsi[0], si[3]))
        dh_ref = da_ref * ogelu.gelu_grad(hq[rows])
        assert rel_fro(dhd[rows], dh_ref) < 2e-3
        dhq = host(g.dhq)
        assert np.array_equal(dhq, ofp8.quantize(dhd, gsc[1], gfmt))
        assert am_b[1] == ofp8.amax(dhd)
        if sample_rows is None:
            dw2_ref = ofp8.decode(dyq, gfmt).T @ ofp8.decode(aq, ffmt) * np.float64(dequant_scale(gsi[0], si[2]))
            assert rel_fro(host(g.dw2), _bf16(dw2_ref)) < 1e-3
            dw1_ref = ofp8.decode(dhq, gfmt).T @ ofp8.decode(lnq, ffmt) * np.float64(dequant_scale(gsi[1], si[0]))
            assert rel_fro(host(g.dw1), _bf16(dw1_ref)) < 1e-3
            assert rel_fro(host(g.db1), dhd.astype(np.float64).sum(axis=0)) < 1e-4
        dln_ref = ofp8.decode(dhq[rows], gfmt) @ ofp8.decode(w1q, ffmt) * np.float64(dequant_scale(gsi[1], si[1]))
        assert rel_fro(host(g.dln)[rows], _bf16(dln_ref)) < 1e-3

        # ---- end to end against the independent oracle (same inputs, same pre-step state)
        fo, bo = fpre.copy(), bpre.copy()
        Y, octx, aux = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fo, orec)
        og = omod.ln_mlp_bwd(dy, octx, bo, orec)
        assert rel_fro(yv, Y) < TOL
        for k in ("dx", "dw1", "dw2", "db1", "db2", "dgamma", "dbeta"):
            gv = host(getattr(g, k))
            assert rel_fro(gv, og[k]) < TOL, (step, k, rel_fro(gv, og[k]))
        # independent amaxes of computed tensors
        assert _rel_amax(am_f[0], ofp8.amax(aux["y"])) < 2e-3
        assert _rel_amax(am_f[2], ofp8.amax(aux["a"])) < TOL
        assert _rel_amax(am_b[1], ofp8.amax(og["dh"])) < TOL
        # the oracle's own state machine agrees on the exact-input slots
        for i in (1, 3):
            assert fo.scale[i] == host(fm.scale)[i]
        assert bo.scale[0] == host(bm.scale)[0]
    return fm, bm


def test_mlp_small_multistep_hybrid(L):
    run_mlp(L, M=300, D=256, F=512, steps=4, hist=3)


def test_mlp_e4m3_format_and_t3_inputs(L):
    run_mlp(L, M=200, D=128, F=384, steps=3, fmt="e4m3", hist=2, dist="t3")


def test_mlp_e5m2_format(L):
    run_mlp(L, M=130, D=128, F=256, steps=2, fmt="e5m2", hist=16, dist="normal")


def test_mlp_without_bias_and_single_row(L):
    run_mlp(L, M=1, D=64, F=128, steps=2, bias_std=0.0)


def test_mlp_empty_batch(L):
    rec = L.Recipe("hybrid", 4)
    D, F = 64, 128
    p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, seed=3).items()}
    fm, bm = L.ScalingMeta(4, 4), L.ScalingMeta(2, 4)
    x = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    y, ctx = L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fm, rec)
    g = L.ln_mlp_bwd(torch.empty(0, D, dtype=torch.bfloat16, device="cuda"), x, p["gamma"], ctx, bm, rec)
    L.sync_status()
    assert y.shape == (0, D)
    for t in (g.dw1, g.dw2, g.db1, g.db2, g.dgamma, g.dbeta):
        assert (host(t) == 0).all()
    am = host(fm.amax_history)[0]
    assert am[0] == 0 and am[2] == 0 and am[1] > 0 and am[3] > 0


def test_mlp_config2_full_size_two_steps(L):
    # LayerNormMLP 768 -> 3072 -> 768 over 8192 tokens (32 x 256), HYBRID, history 16
    run_mlp(L, M=8192, D=768, F=3072, steps=2, hist=16, bias_std=0.0, seed=1234)


def test_mlp_config2_twenty_steps_state(L):
    # the 20-step run of the same workload: state bit-exact (teacher-forced) every step,
    # full parity on the first and last step
    run_mlp(L, M=8192, D=768, F=3072, steps=20, hist=16, bias_std=0.0, seed=1234, full_check_steps={0, 19},
            sample_rows=np.arange(0, 8192, 37))


def test_mlp_d2048_sampled_rows(L):
    # LayerNormMLP 2048 -> 8192 -> 2048 over 2048 tokens, history 1024
    run_mlp(L, M=2048, D=2048, F=8192, steps=2, hist=1024, bias_std=0.0, seed=1234, dist="t3",
            sample_rows=np.arange(0, 2048, 17))


# ------------------------------------------------------------------ LayerNormLinear / Linear
def run_linear(L, M, K, N, steps, ln=True, fmt="hybrid", hist=16, bias_std=0.02, seed=21, path=0):
    rec = L.Recipe(fmt, hist)
    orec = ORecipe(fmt, hist)
    p = synth.linear_params(N, K, ln=ln, bias_std=bias_std, seed=seed)
    w, b = bf16_dev(p["w"]), bf16_dev(p["b"])
    gma = bf16_dev(p["gamma"]) if ln else None
    bta = bf16_dev(p["beta"]) if ln else None
    fm, bm = L.ScalingMeta(2, hist), L.ScalingMeta(1, hist)
    ffmt, gfmt = orec.fwd_fmt(), orec.bwd_fmt()
    for step in range(steps):
        x = synth.activations(M, K, dist="outliers", seed=seed, step=step)
        dy = synth.grad(M, N, seed=seed, step=step)
        xt = bf16_dev(x)
        fpre, bpre = _state_from_gpu(fm), _state_from_gpu(bm)
        y, ctx = L.ln_linear_fwd(xt, gma, bta, w, b, fm, rec, debug=ln, path=path)
        g = L.ln_linear_bwd(bf16_dev(dy), xt, gma, ctx, bm, rec)
        L.sync_status()
        _assert_state_equal(fm, _teacher_forced(fpre, fm, [ffmt] * 2), f"fwd {step}")
        _assert_state_equal(bm, _teacher_forced(bpre, bm, [gfmt]), f"bwd {step}")
        xq = host(ctx.xq)
        if ln:
            ydbg = host(ctx.ln_out_debug)
            assert np.array_equal(xq, ofp8.quantize(ydbg, fpre.scale[0], ffmt))
        else:
            assert np.array_equal(xq, ofp8.quantize(bf16_to_f32(x), fpre.scale[0], ffmt))
        assert np.array_equal(host(ctx.wq), ofp8.quantize(bf16_to_f32(p["w"]), fpre.scale[1], ffmt))
        fo, bo = fpre.copy(), bpre.copy()
        Y, octx, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], fo, orec)
        og = omod.ln_linear_bwd(dy, octx, bo, orec)
        assert rel_fro(host(y), Y) < TOL
        assert rel_fro(host(g.dx), og["dx"]) < TOL
        assert rel_fro(host(g.dw), og["dw"]) < TOL
        assert rel_fro(host(g.dbias), og["db"]) < 1e-4
        if ln:
            assert rel_fro(host(g.dgamma), og["dgamma"]) < TOL
            assert rel_fro(host(g.dbeta), og["dbeta"]) < TOL
    return fm, bm


@pytest.mark.parametrize("path", [1, 2])
def test_linear_config1_qkv_forward_e4m3(L, path):
    # LayerNormLinear 768 -> 2304 over 256 tokens (8 x 32), E4M3, history 16, one step, bias 0;
    # the one-launch fused forward (path 1) and the separate launches (path 2)
    run_linear(L, M=256, K=768, N=2304, steps=1, fmt="e4m3", bias_std=0.0, seed=1234, path=path)


@pytest.mark.parametrize("path", [1, 2])
def test_linear_small_multistep_both_paths(L, path):
    run_linear(L, M=100, K=192, N=400, steps=3, hist=2, path=path)
    run_linear(L, M=70, K=256, N=128, steps=2, ln=False, path=path)


def test_linear_with_ln_multistep_ragged(L):
    run_linear(L, M=333, K=192, N=400, steps=3, hist=2)


def test_linear_without_ln(L):
    run_linear(L, M=250, K=256, N=128, steps=2, ln=False)


@pytest.mark.parametrize("M,ln", [(256, True), (333, True), (0, True), (250, False)])
def test_linear_forward_state_update_in_the_gemm_launch(L, M, ln):
    """With the LayerNorm, the separate-launch forward is two launches: the LayerNorm (with
    the weight cast and the scale_inv snapshot) and the GEMM, whose extra cluster runs the
    state update. Over three steps its outputs and state equal, bit for bit, a deferred
    forward followed by the standalone update; the saved scale_inv is the state's before
    the call. Without the LayerNorm: input cast, weight cast, GEMM, state update."""
    K, N = 768, 2304
    rec = L.Recipe("hybrid", 16)
    p = synth.linear_params(N, K, ln=ln, layer=2, bias_std=0.02)
    dev = {k: bf16_dev(v) for k, v in p.items() if v is not None}
    g, b = (dev["gamma"], dev["beta"]) if ln else (None, None)
    runs = []
    for carried in (True, False):
        meta, ys = L.ScalingMeta(2, 16), []
        for step in range(3):
            x = bf16_dev(synth.activations(M, K, dist="outliers", seed=11, step=step)) if M else \
                torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
            pre = meta.scale_inv.clone()
            n0 = L.launch_count()
            y, ctx = L.ln_linear_fwd(x, g, b, dev["w"], dev["b"], meta, rec, path=L.PATH_SEPARATE,
                                     defer_update=not carried)
            launches = L.launch_count() - n0
            if carried and M > 0:
                assert launches == (2 if ln else 4), launches
            if not carried:
                L.amax_history_update(meta, rec, [L.E4M3, L.E4M3])
            L.sync_status()
            assert torch.equal(ctx.sinv_saved, pre), step
            ys.append(y.clone())
        runs.append((ys, meta))
    (ya, ma), (yb, mb) = runs
    for step in range(3):
        assert torch.equal(ya[step], yb[step]), step
    for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
        assert torch.equal(getattr(ma, name), getattr(mb, name)), name


def test_mlp_step_replayed_from_a_cuda_graph_matches_direct_calls_and_is_profiled(L):
    """The step captured into a CUDA graph (as the benchmark replays it) gives the
    direct call's results; per-kernel timing works for direct calls and for
    replays of a graph captured with timing on."""
    M, D, F = 1000, 256, 1024
    p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, bias_std=0.02, seed=5).items()}
    x = bf16_dev(synth.activations(M, D, dist="outliers", seed=5, step=0))
    dy = bf16_dev(synth.grad(M, D, seed=5, step=0))
    rec = L.Recipe("hybrid", 4)

    def make():
        return L.ScalingMeta(4, 4), L.ScalingMeta(2, 4), L.mlp_ctx(M, D, F), L.mlp_grads(M, D, F)

    def call(fm, bm, ctx, g, y):
        L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fm, rec, y=y, ctx=ctx)
        L.ln_mlp_bwd(dy, x, p["gamma"], ctx, bm, rec, grads=g)

    fm0, bm0, ctx0, g0 = make()
    y0 = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    L.profile_enable(True)
    call(fm0, bm0, ctx0, g0, y0)
    direct = L.profile_collect()
    L.profile_enable(False)
    L.sync_status()
    # forward: LayerNorm with the weight casts and the scale_inv snapshot in the same launch, FC1, FC2 with
    # the state update in an extra cluster; backward: clears, dY cast, the FC2 data and weight gradients in
    # one launch, the FC1 data and weight gradients in one launch, LayerNorm with the state update in extra
    # CTAs of the same launch
    assert sum(n for _, n in direct.values()) == 8 and all(ms > 0 for ms, _ in direct.values())
    assert direct["ln_bwd"][1] == 1 and "state_update" not in direct and "cast_pair" not in direct

    fm1, bm1, ctx1, g1 = make()
    y1 = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    L.profile_enable(True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(fm1, bm1, ctx1, g1, y1)
    graph.replay()
    torch.cuda.synchronize()
    L.profile_sample()
    replayed = L.profile_collect()
    L.profile_enable(False)
    L.sync_status()
    assert set(replayed) == set(direct)
    assert all(replayed[k][1] == direct[k][1] and replayed[k][0] > 0 for k in direct)

    for a, b in [(y0, y1), (g0.dx, g1.dx), (g0.dw1, g1.dw1), (g0.dw2, g1.dw2)]:
        assert torch.equal(a, b)
    for a, b in [(g0.db1, g1.db1), (g0.db2, g1.db2), (g0.dgamma, g1.dgamma), (g0.dbeta, g1.dbeta)]:
        assert rel_fro(host(a), host(b)) < 1e-5  # column sums use float atomics (order may differ)
    for m0, m1 in [(fm0, fm1), (bm0, bm1)]:
        for name in ("scale", "scale_inv", "amax_history"):
            assert torch.equal(getattr(m0, name), getattr(m1, name)), name


@pytest.mark.parametrize("M,D,F", [(8192, 768, 3072), (1000, 256, 1024)])
def test_mlp_backward_split_k_is_deterministic_and_matches_unsplit(L, M, D, F):
    """The backward GEMMs share one split-K workspace, one after another. Two runs
    with it give identical bits, and the same results as the unsplit GEMMs up to
    fp32 summation order (a bf16 ulp on a few elements)."""
    p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, bias_std=0.02, seed=3).items()}
    x = bf16_dev(synth.activations(M, D, dist="outliers", seed=3, step=0))
    dy = bf16_dev(synth.grad(M, D, seed=3, step=0))
    rec = L.Recipe("hybrid", 4)
    ctx = L.mlp_ctx(M, D, F)
    L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], L.ScalingMeta(4, 4), rec, ctx=ctx)
    runs = []
    for split in (True, True, False):
        g = L.mlp_grads(M, D, F, split_k=split)
        assert (g.gemm_ws is not None) == (split and L.ln_mlp_bwd_workspace_size(M, D, F) > 0)
        L.ln_mlp_bwd(dy, x, p["gamma"], ctx, L.ScalingMeta(2, 4), rec, grads=g)
        L.sync_status()
        runs.append(g)
    names = ("dx", "dw1", "dw2", "dln", "dgamma", "dbeta", "db1", "db2")
    for k in ("dx", "dw1", "dw2", "dln"):
        assert torch.equal(getattr(runs[0], k), getattr(runs[1], k)), k
    for k in names:
        a, b = host(getattr(runs[0], k)), host(getattr(runs[2], k))
        assert rel_fro(a, b) < 1e-4, (k, rel_fro(a, b))
    for k in ("dw1", "dw2", "dln"):
        a, b = host(getattr(runs[0], k)), host(getattr(runs[2], k))
        assert np.abs(a - b).max() <= 2.0 ** -7 * np.abs(b).max(), k


@pytest.mark.parametrize("M,D,F", [(8192, 768, 3072), (1008, 256, 1024), (2064, 384, 1552)])
def test_mlp_backward_fc2_weight_gradient_equals_the_standalone_gemm(L, M, D, F):
    """The FC2 weight gradient runs in one launch with the FC2 data gradient. Without a
    split-K workspace its K range is not cut, so it must equal, bit for bit, the
    standalone GEMM of the same codes and scales: dW2 = (dYq^T . Aq) * gsinv[0] * sinv[2]."""
    p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, bias_std=0.02, seed=9).items()}
    x = bf16_dev(synth.activations(M, D, dist="outliers", seed=9, step=0))
    dy = bf16_dev(synth.grad(M, D, seed=9, step=0))
    rec = L.Recipe("hybrid", 4)
    ctx = L.mlp_ctx(M, D, F)
    L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], L.ScalingMeta(4, 4), rec, ctx=ctx)
    bm = L.ScalingMeta(2, 4)
    gsinv = bm.scale_inv.clone()  # the backward state before the call (its update runs at the end)
    g = L.mlp_grads(M, D, F, split_k=False)
    L.ln_mlp_bwd(dy, x, p["gamma"], ctx, bm, rec, grads=g)
    ref = L.fp8_gemm(g.dyq, 1, L.E5M2, ctx.aq, 1, L.E4M3, D, F, M, gsinv[0:1], ctx.sinv_saved[2:3])
    L.sync_status()
    assert torch.equal(g.dw2, ref)


@pytest.mark.parametrize("M,D,F", [(8192, 768, 3072), (1000, 256, 1024), (16, 128, 384)])
def test_mlp_forward_fused_launch_equals_two_launches(L, M, D, F):
    """With its readiness-counter workspace the forward runs FC1 (+GELU) and FC2 as one
    launch, FC2 tiles starting as the FC1 tiles of their rows finish. The arithmetic
    is the same as two launches: Y, H, the GELU codes and the state match bit for bit."""
    p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, bias_std=0.02, seed=4).items()}
    rec = L.Recipe("hybrid", 4)
    outs = []
    for fused in (True, False, True):
        fm = L.ScalingMeta(4, 4)
        ctx = L.mlp_ctx(M, D, F, fused=fused)
        assert (ctx.gemm_ws is not None) == fused
        for step in range(2):  # the second step casts with scales from the first
            x = bf16_dev(synth.activations(M, D, dist="outliers", seed=4, step=step))
            y, _ = L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fm, rec, ctx=ctx)
        L.sync_status()
        outs.append((y, ctx, fm))
    for (y0, c0, m0), (y1, c1, m1) in [(outs[0], outs[1]), (outs[0], outs[2])]:
        assert torch.equal(y0, y1)
        assert torch.equal(c0.h, c1.h) and torch.equal(c0.aq, c1.aq)
        for name in ("scale", "scale_inv", "amax_history"):
            assert torch.equal(getattr(m0, name), getattr(m1, name)), name


@pytest.mark.parametrize("M", [0, 1, 300])
def test_forward_weight_casts_in_the_layernorm_launch(L, M):
    """The forward's weight casts run inside its LayerNorm launch: W1, W2 (LayerNormMLP)
    and W (LayerNormLinear) codes equal the oracle's cast bit for bit, and their amaxes
    reach the history, also with no tokens at all (the launch then only casts) and with
    one token (the grid is sized by the weight tiles). The widths leave ragged 128 x 64
    weight tiles (272 = 4 x 64 + 16 columns, 1040 = 8 x 128 + 16 rows)."""
    D, F, N = 272, 1040, 784
    rec, orec = L.Recipe("hybrid", 4), ORecipe("hybrid", 4)
    ffmt = orec.fwd_fmt()
    p = synth.mlp_params(D, F, seed=17, bias_std=0.02)
    lw = synth.weight(N, D, seed=17, tid=synth.TID["w1"], layer=1)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    fm, lm = L.ScalingMeta(4, 4), L.ScalingMeta(2, 4)
    W1, W2, LW = bf16_to_f32(p["w1"]), bf16_to_f32(p["w2"]), bf16_to_f32(lw)
    for step in range(2):
        fpre, lpre = _state_from_gpu(fm), _state_from_gpu(lm)
        x = bf16_dev(synth.activations(M, D, dist="outliers", seed=17, step=step)) if M else \
            torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
        _, ctx = L.ln_mlp_fwd(x, dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm, rec)
        _, lctx = L.ln_linear_fwd(x, dev["gamma"], dev["beta"], bf16_dev(lw), None, lm, rec)
        L.sync_status()
        assert np.array_equal(host(ctx.w1q), ofp8.quantize(W1, fpre.scale[1], ffmt)), step
        assert np.array_equal(host(ctx.w2q), ofp8.quantize(W2, fpre.scale[3], ffmt)), step
        assert np.array_equal(host(lctx.wq), ofp8.quantize(LW, lpre.scale[1], ffmt)), step
        fh, lh = host(fm.amax_history)[0], host(lm.amax_history)[0]
        assert fh[1] == ofp8.amax(W1) and fh[3] == ofp8.amax(W2) and lh[1] == ofp8.amax(LW), step
        _assert_state_equal(fm, _teacher_forced(fpre, fm, [ffmt] * 4), f"fwd step {step}")
        _assert_state_equal(lm, _teacher_forced(lpre, lm, [ffmt] * 2), f"linear step {step}")
        if M == 0:
            assert fh[0] == 0 and fh[2] == 0 and lh[0] == 0  # no rows: no activation amax
