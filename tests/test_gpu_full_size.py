"""Parity at the benchmarked sizes (GPU), on sampled outputs the oracle computes
one by one.

The benchmark times LayerNormMLP 2048 -> 8192 -> 2048 over 16384 tokens, the
12-layer block stack of that width with history 1024, and the format / size
sweep up to 65536 tokens (TE tutorial, code blocks 4-5: D_MODEL 2048,
N_LAYERS 12, amax_history_len 1024, "Format.E4M3 vs HYBRID"). At those sizes
the GEMMs walk their output tiles in several raster groups (csrc/gemm.cu,
tile_mn: as many 256-row panels per group as fit in 48 MB of L2, 24 at K =
8192), an order no smaller test reaches.

A full oracle step is too slow there, so these tests rest on two exact
separations of the method (pinned on the CPU by tests/test_oracle_sampling.py):
  * given the step's scales, every output row of a module (Y, H, the GELU
    output, dH, dLN, dX) depends only on the same row of its inputs: the oracle
    run on a sample of token rows gives those rows exactly;
  * every FFN column f of a LayerNormMLP (H[:, f], the GELU output and its
    codes, dH[:, f], db1[f], dW1[f, :], dW2[:, f]) depends only on W1[f, :],
    b1[f], W2[:, f] and all tokens, and every output feature n of a
    LayerNormLinear (Y[:, n], dW[n, :], db[n]) only on W[n, :], b[n] and
    dY[:, n]: the oracle run with those weight slices gives them exactly.
The sampled rows take one row from every 128-row block and the sampled columns
one column from every 128-column block, so every output tile of every GEMM is
compared. After every step the state is checked bit for bit against the
oracle's state machine fed the amaxes the GPU recorded, the amaxes of exact
inputs (weights, dY) bit for bit against the oracle's, and the codes of the
fused casts bit for bit against the oracle's cast of the kernel's own fp32
values. Tolerances as elsewhere: 1e-2 relative Frobenius for bf16 outputs and
gradients, 2e-3 for the LayerNorm output.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8 as ofp8
from oracle import gemm as ogemm
from oracle import layernorm as oln
from oracle import modules as omod
from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
from oracle.gemm import bf16_to_f32, to_bf16_bits
from helpers import bf16_dev, host, rel_fro
from oracle import gelu as ogelu
from oracle_pool import draw, mlp_column_run, pquantize, stack_layer_params

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2
LN_TOL = 2e-3


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


@pytest.fixture(scope="module")
def pool():
    # spawn: this process already holds a CUDA context, which a forked worker would inherit
    p = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    yield p
    p.close()
    p.join()


# ------------------------------------------------------------------ helpers
def sample_blocks(n, block=128, salt=0):
    """One index from every block of `block` consecutive indices, at an offset that
    walks through the block (so the samples meet every lane / column position)."""
    out = []
    for b in range((n + block - 1) // block):
        width = min(block, n - b * block)
        out.append(b * block + (b * 37 + salt) % width)
    return np.array(out, dtype=np.int64)


def _rows(t, idx):
    return t.index_select(0, torch.from_numpy(idx).to(t.device))


def _cols(t, idx):
    return t.index_select(1, torch.from_numpy(idx).to(t.device))


def _state(meta):
    s = ScalingState(meta.n, meta.history_len)
    s.scale[:] = host(meta.scale)
    s.scale_inv[:] = host(meta.scale_inv)
    s.amax_history[:] = host(meta.amax_history)
    s.amax_cur[:] = host(meta.amax_cur)
    return s


def _teacher_forced(pre, meta, fmts):
    """The oracle state machine run from the pre-step state with the amaxes the GPU recorded."""
    st = pre.copy()
    am = host(meta.amax_history)[0].astype(np.float32)
    for i in range(st.n):
        st.record(i, am[i])
    st.update(fmts)
    return st


def _assert_state_equal(meta, ost, what):
    for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
        g = host(getattr(meta, name)).astype(np.float32)
        assert np.array_equal(g.view(np.uint32), getattr(ost, name).view(np.uint32)), (what, name)


def _rel_amax(a, b):
    return abs(float(a) - float(b)) / max(abs(float(b)), 1e-30)


def _f64(bits):
    return bf16_to_f32(bits).astype(np.float64)


def to_bits(values):
    return to_bf16_bits(np.asarray(values, np.float64))


# ------------------------------------------------------------------ GEMM: several raster groups
_INT_VALUES = np.arange(-4, 5, dtype=np.float32)


def _int_codes(shape, fmt, rng):
    """Codes of small integers (exact in E4M3 and E5M2): every fp32 sum of products stays exact."""
    return ofp8.encode(_INT_VALUES, fmt)[rng.integers(0, len(_INT_VALUES), size=shape)]


@pytest.mark.parametrize("M,N,K,layouts", [
    (16384, 2048, 8192, [(0, 0), (0, 1), (1, 1), (1, 0)]),  # FC2 / FC1 dgrad at d 2048: 64 row pairs, groups 24+24+16
    (16400, 2064, 8208, [(0, 0), (0, 1), (1, 1), (1, 0)]),  # ragged M, N, K: 65 row pairs, groups 23+23+19
    (8192, 2048, 16384, [(1, 1), (0, 0)]),                   # FC1 weight gradient over 16384 tokens: groups 12+12+8
])
def test_gemm_exact_integer_problems_over_several_raster_groups(L, M, N, K, layouts):
    rng = np.random.default_rng(M + N + K)
    a = _int_codes((M, K), ofp8.E4M3, rng)
    b = _int_codes((N, K), ofp8.E5M2, rng)
    bias = synth.f32_to_bf16_bits(rng.integers(-8, 8, N).astype(np.float32))
    ref = ogemm.fp8_gemm(a, ofp8.E4M3, b, ofp8.E5M2, 0.25, 0.5, bf16_to_f32(bias))
    want = ogemm.bf16_to_f32(ogemm.to_bf16_bits(ref))
    del ref
    s_a = torch.tensor([0.25], device="cuda")
    s_b = torch.tensor([0.5], device="cuda")
    for al, bl in layouts:
        at = torch.from_numpy(np.ascontiguousarray(a if al == 0 else a.T)).cuda()
        bt = torch.from_numpy(np.ascontiguousarray(b if bl == 0 else b.T)).cuda()
        out = L.fp8_gemm(at, al, L.E4M3, bt, bl, L.E5M2, M, N, K, s_a, s_b, bias=bf16_dev(bias))
        got = out.float().cpu().numpy()
        assert np.array_equal(got, want), (al, bl, int((got != want).sum()))
        del at, bt, out


# ------------------------------------------------------------------ LayerNormMLP
def check_mlp_step(L, pool, p, x, dy, fpre, bpre, fm, bm, ctx, g, y, orec, rows, cols, tag):
    """One LayerNormMLP fwd+bwd step of the GPU (outputs y, saved ctx, grads g, debug
    dumps on) against the oracle on sampled rows and FFN columns."""
    ffmt, gfmt = orec.fwd_fmt(), orec.bwd_fmt()
    _assert_state_equal(fm, _teacher_forced(fpre, fm, [ffmt] * 4), tag + " fwd state")
    _assert_state_equal(bm, _teacher_forced(bpre, bm, [gfmt] * 2), tag + " bwd state")
    am_f, am_b = host(fm.amax_history)[0], host(bm.amax_history)[0]
    assert am_f[1] == ofp8.amax(bf16_to_f32(p["w1"])) and am_f[3] == ofp8.amax(bf16_to_f32(p["w2"])), tag
    assert am_b[0] == ofp8.amax(bf16_to_f32(dy)), tag
    sc, si, gsc = fpre.scale, fpre.scale_inv, bpre.scale
    assert np.array_equal(host(ctx.sinv_saved).astype(np.float32).view(np.uint32), si.view(np.uint32)), tag

    # the column run (all tokens, sampled FFN columns) in a worker while the rest is checked here
    w1q_c = ofp8.quantize(bf16_to_f32(p["w1"][cols]), sc[1], ffmt)
    w2q_c = ofp8.quantize(bf16_to_f32(np.ascontiguousarray(p["w2"][:, cols])), sc[3], ffmt)
    col_job = pool.apply_async(mlp_column_run, ((x, dy, p, cols, w1q_c, w2q_c, fpre, bpre, orec),))

    # weight codes: exact inputs, the oracle's cast over the pool
    w1q = pquantize(pool, p["w1"], sc[1], ffmt)
    w2q = pquantize(pool, p["w2"], sc[3], ffmt)
    assert np.array_equal(host(ctx.w1q), w1q) and np.array_equal(host(ctx.w2q), w2q), tag
    assert np.array_equal(w1q[cols], w1q_c) and np.array_equal(w2q[:, cols], w2q_c), tag
    fw = ((w1q, si[1]), (w2q, si[3]))

    # ---- sampled token rows, all columns
    ri = rows
    Yr, ocr, auxr = omod.ln_mlp_fwd(x[ri], p["gamma"], p["beta"], None, p["b1"], None, p["b2"], fpre.copy(), orec,
                                    fp8_weights=fw)
    ogr = omod.ln_mlp_bwd(dy[ri], ocr, bpre.copy(), orec)
    assert rel_fro(host(_rows(y, ri)), Yr) < TOL, tag + " Y rows"
    h_r = host(_rows(ctx.h, ri))
    assert rel_fro(h_r, auxr["h"]) < TOL, tag + " H rows"
    dh_r = host(_rows(g.dh_debug, ri))
    assert rel_fro(dh_r, ogr["dh"]) < TOL, tag + " dH rows"
    assert rel_fro(host(_rows(g.dln, ri)), ogr["dln"]) < TOL, tag + " dLN rows"
    assert rel_fro(host(_rows(g.dx, ri)), ogr["dx"]) < TOL, tag + " dX rows"

    # ---- codes of the fused casts: bit-exact on the kernel's own fp32 values (rows and columns)
    ydbg = host(ctx.ln_out_debug)
    assert am_f[0] == ofp8.amax(ydbg), tag
    assert np.array_equal(host(_rows(ctx.lnq, ri)), ofp8.quantize(ydbg[ri], sc[0], ffmt)), tag + " LN codes"
    a_r, a_c = host(_rows(ctx.act_debug, ri)), host(_cols(ctx.act_debug, cols))
    dh_c = host(_cols(g.dh_debug, cols))
    assert np.array_equal(host(_rows(ctx.aq, ri)), ofp8.quantize(a_r, sc[2], ffmt)), tag + " A codes rows"
    assert np.array_equal(host(_cols(ctx.aq, cols)), ofp8.quantize(a_c, sc[2], ffmt)), tag + " A codes columns"
    assert np.array_equal(host(_rows(g.dhq, ri)), ofp8.quantize(dh_r, gsc[1], gfmt)), tag + " dH codes rows"
    assert np.array_equal(host(_cols(g.dhq, cols)), ofp8.quantize(dh_c, gsc[1], gfmt)), tag + " dH codes columns"
    # the kernel's GELU output against the oracle's GELU of the kernel's own bf16 H
    assert np.abs(a_r - ogelu.gelu(h_r)).max() <= LN_TOL * np.abs(a_r).max(), tag + " GELU"
    # the amaxes of the computed tensors are the max of the kernel's own values
    assert am_f[2] == ofp8.amax(host(ctx.act_debug)), tag
    assert am_b[1] == ofp8.amax(host(g.dh_debug)), tag

    # ---- LayerNorm parameter gradients: the oracle's LayerNorm backward of the kernel's dLN
    _, dg_ref, db_ref = oln.backward(host(g.dln), _f64(x), _f64(p["gamma"]))
    assert rel_fro(host(g.dgamma), dg_ref) < TOL, tag + " dgamma"
    assert rel_fro(host(g.dbeta), db_ref) < TOL, tag + " dbeta"

    # ---- sampled FFN columns, all tokens (the column run)
    oc = col_job.get()
    h_c = host(_cols(ctx.h, cols))
    assert rel_fro(h_c, oc["h"]) < TOL, tag + " H columns"
    assert rel_fro(dh_c, oc["dh"]) < TOL, tag + " dH columns"
    assert rel_fro(host(g.db1)[cols], oc["db1"]) < TOL, tag + " db1"
    assert rel_fro(host(_rows(g.dw1, cols)), oc["dw1"]) < TOL, tag + " dW1 rows"
    assert rel_fro(host(_cols(g.dw2, cols)), oc["dw2"]) < TOL, tag + " dW2 columns"
    assert rel_fro(host(g.db2), oc["db2"]) < 1e-4, tag + " db2"
    assert np.array_equal(host(g.dyq), oc["dyq"]), tag + " dY codes"
    # amaxes of the computed tensors: at least the oracle's maximum over the sampled rows and columns
    assert float(am_f[2]) >= (1 - TOL) * max(float(ofp8.amax(auxr["a"])), float(ofp8.amax(oc["a"]))), tag
    assert float(am_b[1]) >= (1 - TOL) * max(float(ofp8.amax(ogr["dh"])), float(ofp8.amax(oc["dh"]))), tag

    # ---- LayerNorm output of all tokens (the column run normalises every row)
    assert np.abs(ydbg - oc["y"]).max() <= LN_TOL * max(1.0, np.abs(oc["y"]).max()), tag + " LN"
    assert _rel_amax(am_f[0], ofp8.amax(oc["y"])) < LN_TOL, tag


def run_mlp_sampled(L, pool, M, D, F, steps, fmt, hist, dist, seed, bias_std=0.02):
    rec, orec = L.Recipe(fmt, hist), ORecipe(fmt, hist)
    p = synth.mlp_params(D, F, seed=seed, bias_std=bias_std)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    fm, bm = L.ScalingMeta(4, hist), L.ScalingMeta(2, hist)
    ctx = L.mlp_ctx(M, D, F, debug=True)
    g = L.mlp_grads(M, D, F, debug=True)  # with the split-K workspace, as the benchmark runs it
    y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    rows, cols = sample_blocks(M, salt=seed), sample_blocks(F, salt=seed + 1)
    for step in range(steps):
        x, dy = pool.map(draw, [("act", M, D, dict(dist=dist, seed=seed, step=step)),
                                            ("grad", M, D, dict(seed=seed, step=step))])
        xt, dyt = bf16_dev(x), bf16_dev(dy)
        fpre, bpre = _state(fm), _state(bm)
        L.ln_mlp_fwd(xt, dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm, rec, y=y, ctx=ctx)
        L.ln_mlp_bwd(dyt, xt, dev["gamma"], ctx, bm, rec, grads=g)
        L.sync_status()
        check_mlp_step(L, pool, p, x, dy, fpre, bpre, fm, bm, ctx, g, y, orec, rows, cols,
                       f"{M}x{D}x{F} {fmt} {dist} L{hist} step {step}")
        del xt, dyt


def test_mlp_d2048_16384_tokens_two_steps(L, pool):
    # the benchmark's d 2048 LayerNormMLP: FC2 and the FC1 data-gradient pair walk three raster groups
    run_mlp_sampled(L, pool, 16384, 2048, 8192, steps=2, fmt="hybrid", hist=1024, dist="outliers", seed=1234)


@pytest.mark.parametrize("M,fmt,dist,hist", [
    (32768, "e4m3", "t3", 16),
    (32768, "hybrid", "normal", 1024),
    (65536, "hybrid", "t3", 16),
    (65536, "e4m3", "normal", 1024),
])
def test_mlp_d2048_format_size_sweep_points(L, pool, M, fmt, dist, hist):
    # points of the E4M3-vs-HYBRID, N(0,1)-vs-Student-t(3) sweep at 32768 and 65536 tokens
    run_mlp_sampled(L, pool, M, 2048, 8192, steps=1, fmt=fmt, hist=hist, dist=dist, seed=77)


# ------------------------------------------------------------------ LayerNormLinear / Linear
@pytest.mark.parametrize("K,N,ln", [(2048, 6144, True), (2048, 2048, False)])
def test_linear_d2048_16384_tokens_two_steps(L, pool, K, N, ln):
    """The stack's QKV LayerNormLinear 2048 -> 6144 and the projection Linear 2048 -> 2048
    over 16384 tokens, history 1024, on sampled token rows and output features."""
    M, hist, seed = 16384, 1024, 4242
    rec, orec = L.Recipe("hybrid", hist), ORecipe("hybrid", hist)
    ffmt, gfmt = orec.fwd_fmt(), orec.bwd_fmt()
    p = synth.linear_params(N, K, ln=ln, bias_std=0.02, seed=seed)
    w, b = bf16_dev(p["w"]), bf16_dev(p["b"])
    gma = bf16_dev(p["gamma"]) if ln else None
    bta = bf16_dev(p["beta"]) if ln else None
    fm, bm = L.ScalingMeta(2, hist), L.ScalingMeta(1, hist)
    ctx = L.linear_ctx(M, K, N, ln=ln, debug=ln)
    g = L.linear_grads(M, K, N, ln=ln)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    rows, cols = sample_blocks(M, salt=3), sample_blocks(N, salt=5)
    for step in range(2):
        x, dy = pool.map(draw, [("act", M, K, dict(dist="outliers", seed=seed, step=step)),
                                            ("grad", M, N, dict(seed=seed, step=step))])
        xt = bf16_dev(x)
        fpre, bpre = _state(fm), _state(bm)
        L.ln_linear_fwd(xt, gma, bta, w, b, fm, rec, y=y, ctx=ctx)
        L.ln_linear_bwd(bf16_dev(dy), xt, gma, ctx, bm, rec, grads=g)
        L.sync_status()
        tag = f"{K}->{N} ln={ln} step {step}"
        _assert_state_equal(fm, _teacher_forced(fpre, fm, [ffmt] * 2), tag)
        _assert_state_equal(bm, _teacher_forced(bpre, bm, [gfmt]), tag)
        am_f, am_b = host(fm.amax_history)[0], host(bm.amax_history)[0]
        assert am_f[1] == ofp8.amax(bf16_to_f32(p["w"])) and am_b[0] == ofp8.amax(bf16_to_f32(dy)), tag
        sc, si = fpre.scale, fpre.scale_inv
        wq = pquantize(pool, p["w"], sc[1], ffmt)
        assert np.array_equal(host(ctx.wq), wq), tag + " W codes"
        if not ln:  # Linear: the input itself is cast (exact input)
            assert am_f[0] == ofp8.amax(bf16_to_f32(x)), tag
            assert np.array_equal(host(ctx.xq), pquantize(pool, x, sc[0], ffmt)), tag + " X codes"
        # sampled token rows
        Yr, ocr, _ = omod.ln_linear_fwd(x[rows], p["gamma"], p["beta"], None, p["b"], fpre.copy(), orec,
                                        fp8_weight=(wq, si[1]))
        ogr = omod.ln_linear_bwd(dy[rows], ocr, bpre.copy(), orec)
        assert rel_fro(host(_rows(y, rows)), Yr) < TOL, tag + " Y rows"
        assert rel_fro(host(_rows(g.dx, rows)), ogr["dx"]) < TOL, tag + " dX rows"
        # sampled output features, all tokens
        Yc, occ, auxc = omod.ln_linear_fwd(x, p["gamma"], p["beta"], None, p["b"][cols], fpre.copy(), orec,
                                           fp8_weight=(np.ascontiguousarray(wq[cols]), si[1]))
        ogc = omod.ln_linear_bwd(np.ascontiguousarray(dy[:, cols]), occ, bpre.copy(), orec)
        assert rel_fro(host(_cols(y, cols)), Yc) < TOL, tag + " Y columns"
        assert rel_fro(host(_rows(g.dw, cols)), ogc["dw"]) < TOL, tag + " dW rows"
        assert rel_fro(host(g.dbias)[cols], ogc["db"]) < 1e-4, tag + " db"
        assert np.array_equal(host(_cols(g.dyq, cols)), ogc["dyq"]), tag + " dY codes"
        if ln:
            ydbg = host(ctx.ln_out_debug)
            assert np.abs(ydbg - auxc["y"]).max() <= LN_TOL * max(1.0, np.abs(auxc["y"]).max()), tag + " LN"
            assert am_f[0] == ofp8.amax(ydbg) and _rel_amax(am_f[0], ofp8.amax(auxc["y"])) < LN_TOL, tag
            assert np.array_equal(host(_rows(ctx.xq, rows)), ofp8.quantize(ydbg[rows], sc[0], ffmt)), tag
            _, dg_ref, db_ref = oln.backward(host(g.dln), _f64(x), _f64(p["gamma"]))
            assert rel_fro(host(g.dgamma), dg_ref) < TOL and rel_fro(host(g.dbeta), db_ref) < TOL, tag


# ------------------------------------------------------------------ the 12-layer block stack
def test_block_stack_12_layers_d2048_16384_tokens(L, pool):
    """The benchmark's stack step itself (bench.StackRun: every module with its state
    update deferred, one update launch for all 72 state sets, the step replayed as
    one captured CUDA graph), fed seeded host inputs: 12 layers of LayerNormLinear
    2048 -> 6144, Linear 2048 -> 2048 on a synthetic attention output and LayerNormMLP
    2048 -> 8192 -> 2048, chained forward as a pre-LN block (the residual adds fused
    into the next LayerNorm), 16384 tokens, HYBRID, history 1024, three steps; the
    attention output, dQKV and dY are shared by the layers.

    On the sampled rows, every step and layer, from the GPU's pre-step state (which
    is itself checked bit for bit against the oracle's state machine):
      * the oracle's own residual chain from h0 through all layers: the stream
        entering a module sums k terms (h0, then one projection and one MLP output
        per layer), each carrying its own FP8 error within the module bound, so
        the GPU's stream must agree within 1e-2 * sqrt(k);
      * one layer deep, from the GPU's own stream: every module output and input
        gradient within 1e-2, and the fused residual adds bit for bit (the
        oracle's bf16 sum of the GPU's two bf16 tensors)."""
    import bench

    layers, M, D, F, hist, seed = 12, 16384, 2048, 8192, 1024, 99
    rec, orec = L.Recipe("hybrid", hist), ORecipe("hybrid", hist)
    ff, gf = orec.fwd_fmt(), orec.bwd_fmt()
    P = pool.map(stack_layer_params, [(l, D, F, seed, 0.02) for l in range(layers)])
    h0, attn, dqkv, dy = pool.map(draw, [
        ("act", M, D, dict(dist="outliers", seed=seed)),
        ("act", M, D, dict(seed=seed, tid=synth.TID["attn"])),
        ("grad", M, 3 * D, dict(seed=seed, tid=synth.TID["attn"])),
        ("grad", M, D, dict(seed=seed))])
    srun = bench.StackRun(L, torch, torch.device("cuda"), layers, M, D, F, "hybrid", hist, seed=0, host_params=P,
                          host_inputs=dict(h0=h0, attn=attn, dqkv=dqkv, dy=dy), keep_outputs=True)
    srun.capture()
    order = srun.order  # fq fp fm bq bp bm per layer
    ofmts = {"fq": [ff] * 2, "fp": [ff] * 2, "fm": [ff] * 4, "bq": [gf], "bp": [gf], "bm": [gf] * 2}
    rows = sample_blocks(M, salt=11)
    ex = {"attn": ofp8.amax(bf16_to_f32(attn)), "dqkv": ofp8.amax(bf16_to_f32(dqkv)), "dy": ofp8.amax(bf16_to_f32(dy))}
    wam = [{k: ofp8.amax(bf16_to_f32(P[l][k])) for k in ("wqkv", "wproj", "w1", "w2")} for l in range(layers)]
    codes = {}

    def wcodes(l, name, scale):
        key = (l, name, np.float32(scale).tobytes())
        if key not in codes:
            codes[key] = pquantize(pool, P[l][name], scale, ff)
        return codes[key]

    def bits(t):
        return host(_rows(t, rows).view(torch.int16)).view(np.uint16)

    for step in range(3):
        pre = [{k: _state(lay[k]) for k in order} for lay in srun.layer]
        srun.step(step)
        L.sync_status()
        tag = f"step {step}"
        # ---- states: one update launch for all 72 sets, each bit-exact against the oracle rule
        for l, lay in enumerate(srun.layer):
            for k in order:
                _assert_state_equal(lay[k], _teacher_forced(pre[l][k], lay[k], ofmts[k]), (tag, l, k))
            am = {k: host(lay[k].amax_history)[0] for k in order}
            assert am["fq"][1] == wam[l]["wqkv"] and am["fp"][1] == wam[l]["wproj"], (tag, l)
            assert am["fm"][1] == wam[l]["w1"] and am["fm"][3] == wam[l]["w2"], (tag, l)
            assert am["fp"][0] == ex["attn"] and am["bq"][0] == ex["dqkv"], (tag, l)
            assert am["bp"][0] == ex["dy"] and am["bm"][0] == ex["dy"], (tag, l)

        def modules(l, x_bits, res=None, mlp_in=None):
            """The oracle's layer l on the sampled rows: QKV on x (+ res), the projection, and
            the MLP on mlp_in (default: the QKV's stream plus the projection output)."""
            sq, sp, sm = pre[l]["fq"], pre[l]["fp"], pre[l]["fm"]
            Yq, ocq, auxq = omod.ln_linear_fwd(x_bits, P[l]["g1"], P[l]["be1"], None, P[l]["bqkv"], sq.copy(), orec,
                                               fp8_weight=(wcodes(l, "wqkv", sq.scale[1]), sq.scale_inv[1]),
                                               residual=res)
            hq = auxq["x_sum"] if res is not None else _f64(x_bits)
            Yp, ocp, _ = omod.ln_linear_fwd(attn[rows], None, None, None, P[l]["bproj"], sp.copy(), orec,
                                            fp8_weight=(wcodes(l, "wproj", sp.scale[1]), sp.scale_inv[1]))
            fw = ((wcodes(l, "w1", sm.scale[1]), sm.scale_inv[1]), (wcodes(l, "w2", sm.scale[3]), sm.scale_inv[3]))
            if mlp_in is None:
                Ym, ocm, auxm = omod.ln_mlp_fwd(hq, P[l]["g2"], P[l]["be2"], None, P[l]["b1"], None, P[l]["b2"],
                                                sm.copy(), orec, fp8_weights=fw, residual=Yp)
            else:
                Ym, ocm, auxm = omod.ln_mlp_fwd(mlp_in, P[l]["g2"], P[l]["be2"], None, P[l]["b1"], None, P[l]["b2"],
                                                sm.copy(), orec, fp8_weights=fw)
            return dict(Yq=Yq, ocq=ocq, auxq=auxq, hq=hq, Yp=Yp, ocp=ocp, Ym=Ym, ocm=ocm, auxm=auxm)

        def residual_sum(l, a_bits, r_bits):
            """The oracle's fused residual add ahead of a LayerNorm module: bf16(a + r) as bits."""
            sq = pre[l]["fq"]
            aux = omod.ln_linear_fwd(a_bits, P[l]["g1"], P[l]["be1"], None, P[l]["bqkv"], sq.copy(), orec,
                                     fp8_weight=(wcodes(l, "wqkv", sq.scale[1]), sq.scale_inv[1]), residual=r_bits)[2]
            return to_bits(aux["x_sum"])

        # ---- the oracle's own residual chain from h0 (independent of every GPU output)
        xin, res = h0[rows], None
        for l, lay in enumerate(srun.layer):
            o = modules(l, xin, res)
            k_in = 2 * l + 1  # terms summed into the stream entering layer l
            if l > 0:
                assert rel_fro(host(_rows(lay["cq"].x_sum, rows)), o["hq"]) < TOL * np.sqrt(k_in), (tag, l, "stream")
            assert rel_fro(host(_rows(lay["cm"].x_sum, rows)), o["auxm"]["x_sum"]) < TOL * np.sqrt(k_in + 1), \
                (tag, l, "stream into the MLP")
            xin, res = o["auxm"]["x_sum"], o["Ym"]
        # ---- one layer deep, from the GPU's own stream
        for l, lay in enumerate(srun.layer):
            hq_bits = h0[rows] if l == 0 else bits(lay["cq"].x_sum)
            if l > 0:  # the QKV LayerNorm's fused add: x_sum = bf16(previous MLP stream + previous MLP output)
                prev = srun.layer[l - 1]
                assert np.array_equal(residual_sum(l, bits(prev["cm"].x_sum), bits(prev["ym"])), hq_bits), \
                    (tag, l, "fused residual add into QKV")
            xm_bits = bits(lay["cm"].x_sum)
            # the MLP LayerNorm's fused add: x_sum = bf16(stream + projection output), both the GPU's
            assert np.array_equal(residual_sum(l, hq_bits, bits(lay["yp"])), xm_bits), \
                (tag, l, "fused residual add into the MLP")
            o = modules(l, hq_bits, mlp_in=xm_bits)
            assert rel_fro(host(_rows(lay["yq"], rows)), o["Yq"]) < TOL, (tag, l, "QKV output")
            assert rel_fro(host(_rows(lay["yp"], rows)), o["Yp"]) < TOL, (tag, l, "projection output")
            assert rel_fro(host(_rows(lay["ym"], rows)), o["Ym"]) < TOL, (tag, l, "MLP output")
            am = {k: host(lay[k].amax_history)[0] for k in ("fq", "fm", "bm")}
            assert float(am["fq"][0]) >= (1 - LN_TOL) * float(ofp8.amax(o["auxq"]["y"])), (tag, l)
            assert float(am["fm"][0]) >= (1 - LN_TOL) * float(ofp8.amax(o["auxm"]["y"])), (tag, l)
            assert float(am["fm"][2]) >= (1 - TOL) * float(ofp8.amax(o["auxm"]["a"])), (tag, l)
            # backward (not chained: each layer has its own upstream gradients)
            ogm = omod.ln_mlp_bwd(dy[rows], o["ocm"], pre[l]["bm"].copy(), orec)
            assert rel_fro(host(_rows(lay["gm"].dx, rows)), ogm["dx"]) < TOL, (tag, l, "MLP dX")
            assert float(am["bm"][1]) >= (1 - TOL) * float(ofp8.amax(ogm["dh"])), (tag, l)
            ogp = omod.ln_linear_bwd(dy[rows], o["ocp"], pre[l]["bp"].copy(), orec)
            assert rel_fro(host(_rows(lay["gp"].dx, rows)), ogp["dx"]) < TOL, (tag, l, "projection dX")
            ogq = omod.ln_linear_bwd(dqkv[rows], o["ocq"], pre[l]["bq"].copy(), orec)
            assert rel_fro(host(_rows(lay["gq"].dx, rows)), ogq["dx"]) < TOL, (tag, l, "QKV dX")
    del srun
    torch.cuda.empty_cache()
