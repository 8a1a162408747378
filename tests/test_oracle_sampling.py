"""Pins of the two separations the full-size GPU parity tests sample with (CPU).

Given a step's scales, the oracle's LayerNormMLP and LayerNormLinear are
separable:
  * by token row: run on a subset of rows, every row-wise result (Y, H, the
    GELU output, dH and its codes, dLN, dX) equals the full run's rows;
  * by FFN column (LayerNormMLP) or output feature (LayerNormLinear): run with
    the matching slices of the weights and biases (and, for LayerNormLinear, of
    dY), the column-wise results (H, the GELU output and its codes, dH, db1,
    dW1 rows, dW2 columns; Y columns, dW rows, db) equal the full run's.
The weights are passed as the codes of the oracle's own cast (the FP8-weight
branch), cast row slice by row slice as the GPU tests' process pool does; that
branch with those codes is the bf16-weight branch bit for bit. A wrongly
restricted slice (a transposed W2 slice, a dropped bias slice, rows taken from
another step) fails these equalities.
"""
import numpy as np

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8 as ofp8
from oracle import modules as omod
from oracle.delayed_scaling import Recipe, ScalingState
from oracle_pool import quantize_bf16_rows

ROWS = np.array([0, 7, 128, 200, 299])
COLS = np.array([1, 130, 255, 383])


def _split_cast(bits, scale, fmt, parts=3):
    return np.concatenate([quantize_bf16_rows((c, np.float32(scale), fmt))
                           for c in np.array_split(bits, parts, axis=0)], axis=0)


def _eq(a, b):
    return np.array_equal(np.asarray(a), np.asarray(b))


def test_row_split_cast_equals_one_cast():
    w = synth.weight(257, 96, seed=5)
    for scale in (1.0, 3.25, 448.0 / 0.07):
        assert _eq(_split_cast(w, scale, ofp8.E4M3, parts=5), ofp8.quantize(synth.bf16_bits_to_f32(w), scale,
                                                                             ofp8.E4M3))


def _mlp_states(p, rec, M, D, seed):
    """States after one full step, so that the step under test casts with scales other than 1."""
    fs, bs = ScalingState(4, 4), ScalingState(2, 4)
    x = synth.activations(M, D, dist="outliers", seed=seed, step=0)
    dy = synth.grad(M, D, seed=seed, step=0)
    _, c, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs, rec)
    omod.ln_mlp_bwd(dy, c, bs, rec)
    return fs, bs


def test_mlp_separates_by_rows_and_ffn_columns():
    M, D, F, seed = 300, 64, 384, 3
    for fmt in ("hybrid", "e4m3"):
        rec = Recipe(fmt, 4)
        ff = rec.fwd_fmt()
        p = synth.mlp_params(D, F, seed=seed, bias_std=0.02)
        fs, bs = _mlp_states(p, rec, M, D, seed)
        assert fs.scale[0] != 1 and bs.scale[1] != 1
        x = synth.activations(M, D, dist="outliers", seed=seed, step=1)
        dy = synth.grad(M, D, seed=seed, step=1)
        Y, c, aux = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs.copy(), rec)
        g = omod.ln_mlp_bwd(dy, c, bs.copy(), rec)
        w1q, w2q = _split_cast(p["w1"], fs.scale[1], ff), _split_cast(p["w2"], fs.scale[3], ff)
        assert _eq(w1q, c.wq[0]) and _eq(w2q, c.wq[1])
        si = fs.scale_inv
        # token rows
        Yr, cr, ar = omod.ln_mlp_fwd(x[ROWS], p["gamma"], p["beta"], None, p["b1"], None, p["b2"], fs.copy(), rec,
                                     fp8_weights=((w1q, si[1]), (w2q, si[3])))
        gr = omod.ln_mlp_bwd(dy[ROWS], cr, bs.copy(), rec)
        assert _eq(Yr, Y[ROWS])
        for k in ("h", "a", "y"):
            assert _eq(ar[k], aux[k][ROWS]), k
        for k in ("dx", "dh", "dhq", "dln", "dyq"):
            assert _eq(gr[k], g[k][ROWS]), k
        # FFN columns
        _, cc, ac = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], None, p["b1"][COLS], None, p["b2"], fs.copy(), rec,
                                    fp8_weights=((np.ascontiguousarray(w1q[COLS]), si[1]),
                                                 (np.ascontiguousarray(w2q[:, COLS]), si[3])))
        gc = omod.ln_mlp_bwd(dy, cc, bs.copy(), rec)
        for k in ("h", "a"):
            assert _eq(ac[k], aux[k][:, COLS]), k
        assert _eq(ac["y"], aux["y"]) and _eq(cc.aq, c.aq[:, COLS])
        for k in ("dh", "dhq"):
            assert _eq(gc[k], g[k][:, COLS]), k
        assert _eq(gc["dw1"], g["dw1"][COLS]) and _eq(gc["dw2"], g["dw2"][:, COLS])
        assert np.allclose(gc["db1"], g["db1"][COLS], rtol=1e-12, atol=0)
        assert _eq(gc["dyq"], g["dyq"]) and _eq(gc["db2"], g["db2"])


def test_linear_separates_by_rows_and_output_features():
    M, K, N, seed = 300, 64, 384, 8
    for ln in (True, False):
        rec = Recipe("hybrid", 4)
        ff = rec.fwd_fmt()
        p = synth.linear_params(N, K, ln=ln, bias_std=0.02, seed=seed)
        fs, bs = ScalingState(2, 4), ScalingState(1, 4)
        x0 = synth.activations(M, K, dist="outliers", seed=seed, step=0)
        _, c0, _ = omod.ln_linear_fwd(x0, p["gamma"], p["beta"], p["w"], p["b"], fs, rec)
        omod.ln_linear_bwd(synth.grad(M, N, seed=seed, step=0), c0, bs, rec)
        x = synth.activations(M, K, dist="outliers", seed=seed, step=1)
        dy = synth.grad(M, N, seed=seed, step=1)
        Y, c, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], p["w"], p["b"], fs.copy(), rec)
        g = omod.ln_linear_bwd(dy, c, bs.copy(), rec)
        wq = _split_cast(p["w"], fs.scale[1], ff)
        assert _eq(wq, c.wq[0])
        si = fs.scale_inv
        Yr, cr, _ = omod.ln_linear_fwd(x[ROWS], p["gamma"], p["beta"], None, p["b"], fs.copy(), rec,
                                       fp8_weight=(wq, si[1]))
        gr = omod.ln_linear_bwd(dy[ROWS], cr, bs.copy(), rec)
        assert _eq(Yr, Y[ROWS]) and _eq(gr["dx"], g["dx"][ROWS]) and _eq(gr["dyq"], g["dyq"][ROWS])
        Yc, cc, _ = omod.ln_linear_fwd(x, p["gamma"], p["beta"], None, p["b"][COLS], fs.copy(), rec,
                                       fp8_weight=(np.ascontiguousarray(wq[COLS]), si[1]))
        gc = omod.ln_linear_bwd(np.ascontiguousarray(dy[:, COLS]), cc, bs.copy(), rec)
        assert _eq(Yc, Y[:, COLS]) and _eq(gc["dw"], g["dw"][COLS]) and _eq(gc["dyq"], g["dyq"][:, COLS])
        assert np.allclose(gc["db"], g["db"][COLS], rtol=1e-12, atol=0)


def test_a_wrong_slice_is_caught():
    """Planted: W2 sliced by rows instead of columns (shapes made to fit) must not pass."""
    M, D, F, seed = 64, 32, 32, 4
    rec = Recipe("hybrid", 4)
    p = synth.mlp_params(D, F, seed=seed, bias_std=0.02)
    fs, bs = ScalingState(4, 4), ScalingState(2, 4)
    x = synth.activations(M, D, seed=seed)
    dy = synth.grad(M, D, seed=seed)
    _, c, aux = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs.copy(), rec)
    g = omod.ln_mlp_bwd(dy, c, bs.copy(), rec)
    cols = np.array([1, 5, 9])
    w1q, w2q = c.wq
    si = fs.scale_inv
    _, cc, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], None, p["b1"][cols], None, p["b2"], fs.copy(), rec,
                               fp8_weights=((w1q[cols], si[1]), (np.ascontiguousarray(w2q[cols].T), si[3])))
    gc = omod.ln_mlp_bwd(dy, cc, bs.copy(), rec)
    assert not _eq(gc["dh"], g["dh"][:, cols])
