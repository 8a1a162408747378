"""The oracle's pins catch plausible mistakes (CPU only).

Each test plants one mistake in a copy of an oracle function, on the CPU, and
checks that the corresponding pin then fails. Nothing here touches the GPU.
"""
import numpy as np
import pytest

from oracle import fp8, layernorm, modules
from oracle.delayed_scaling import ScalingState
import test_oracle_fp8 as pins_fp8
import test_oracle_state as pins_state
import test_oracle_modules as pins_mod
import test_oracle_numerics as pins_num


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_ties_away_from_zero_is_caught(monkeypatch):
    real = fp8.encode

    def away(x, fmt):  # round half away from zero instead of to even
        x = np.asarray(x, np.float32)
        c = real(x, fmt)
        nxt = np.nextafter(np.abs(x), np.float32(np.inf)).astype(np.float32) * np.where(np.signbit(x), -1, 1)
        c2 = real(nxt.astype(np.float32), fmt)
        vals = np.abs(fp8.decode(c, fmt))
        return np.where(np.abs(x) > vals, c2, c)
    monkeypatch.setattr(fp8, "encode", away)
    cases = [c for c in pins_fp8._golden_cases() if "tie" in c[3]]
    assert any(_fails(pins_fp8.test_hand_worked_cast_cases, *c) for c in cases)


def test_history_rolled_the_wrong_way_is_caught(monkeypatch):
    def bad_update(self, fmts, algo="max", margin=0):
        for i in range(self.n):
            # newest amax written to the last row, oldest dropped from row 0
            self.amax_history[:-1, i] = self.amax_history[1:, i].copy()
            self.amax_history[-1, i] = self.amax_cur[i]
            self.amax_cur[i] = 0
            a = self.amax_history[:, i].max()
            if np.isfinite(a) and a > 0:
                self.scale[i] = np.float32(fp8.FP8_MAX[fmts[i]]) / a
                self.scale_inv[i] = np.float32(1) / self.scale[i]
    monkeypatch.setattr(ScalingState, "update", bad_update)
    assert _fails(pins_state.test_history_row_zero_is_the_latest_step_and_cur_is_cleared)


def test_window_one_step_too_long_is_caught():
    real_L = 2
    fmt, L, am, exp = pins_state._golden()[0]
    st = ScalingState(1, real_L + 1)
    got = []
    for a in am:
        st.record(0, np.float32(a))
        st.update([fmt])
        got.append(float(st.scale[0]))
    assert got != exp


def test_layernorm_backward_without_the_mean_term_is_caught(monkeypatch):
    real = layernorm.backward

    def bad(dy, x, gamma, eps=layernorm.EPS):
        dx, dg, db = real(dy, x, gamma, eps)
        g = np.asarray(dy, np.float64) * np.asarray(gamma, np.float64)[None, :]
        xd = np.asarray(x, np.float64)
        rs = 1 / np.sqrt(xd.var(axis=1) + eps)
        return dx + rs[:, None] * g.mean(axis=1, keepdims=True), dg, db
    monkeypatch.setattr(layernorm, "backward", bad)
    assert _fails(pins_num.test_layernorm_backward_matches_autograd_and_finite_differences)


def test_mlp_wgrad_with_swapped_operands_is_caught(monkeypatch):
    real = modules.ln_mlp_bwd

    def bad(dy, ctx, gstate, recipe, **kw):
        r = real(dy, ctx, gstate, recipe, **kw)
        r["db1"] = r["db1"][::-1].copy()  # bias gradient summed into the wrong columns
        return r
    monkeypatch.setattr(modules, "ln_mlp_bwd", bad)
    assert _fails(pins_mod.test_exact_mlp_equals_fp64_autograd, "tanh")


def test_gelu_on_fp32_h_instead_of_saved_bf16_h_changes_codes():
    # The reading that GELU consumes the saved bf16 H is observable: A computed
    # from the unrounded H gives different E4M3 codes for some entries.
    rng = np.random.default_rng(0)
    h = rng.standard_normal(4096) * 3
    from oracle import gelu as g
    from oracle.gemm import bf16_to_f32, to_bf16_bits
    hb = bf16_to_f32(to_bf16_bits(h)).astype(np.float64)
    c1 = fp8.quantize(g.gelu(hb).astype(np.float32), 1.0, fp8.E4M3)
    c2 = fp8.quantize(g.gelu(h).astype(np.float32), 1.0, fp8.E4M3)
    assert (c1 != c2).any()
