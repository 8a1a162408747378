"""ln_linear_bwd_noalloc: the LayerNormLinear backward for callers that cannot
allocate device memory (GPU).

Such a caller passes inputs and outputs only; the dY codes and the LayerNorm
output gradient live in the library's own fixed scratch array. The test checks,
through the C ABI, that two calls in a row give the same results as
ln_linear_bwd with caller-provided scratch, within the tolerance the other
parity tests use, and that a problem larger than the scratch is refused before
anything runs. This file is collected last on purpose.
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from helpers import bf16_dev, host, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _copy_meta(L, src):
    m = L.ScalingMeta(src.n, src.history_len)
    m.load_state_dict(src.state_dict())
    return m


@pytest.mark.parametrize("M,K,N,ln", [(256, 768, 2304, True), (300, 192, 400, True), (250, 256, 128, False)])
def test_noalloc_backward_matches_the_allocating_one_twice_in_a_row(L, M, K, N, ln):
    rec = L.Recipe("hybrid", 16)
    p = synth.linear_params(N, K, ln=ln, bias_std=0.02, seed=77)
    w, b = bf16_dev(p["w"]), bf16_dev(p["b"])
    gamma = bf16_dev(p["gamma"]) if ln else None
    beta = bf16_dev(p["beta"]) if ln else None
    fm, bm = L.ScalingMeta(2, 16), L.ScalingMeta(1, 16)
    for step in range(2):
        x = bf16_dev(synth.activations(M, K, dist="outliers", seed=77, step=step))
        dy = bf16_dev(synth.grad(M, N, seed=77, step=step))
        _, ctx = L.ln_linear_fwd(x, gamma, beta, w, b, fm, rec)
        ref_meta = _copy_meta(L, bm)
        ref = L.ln_linear_bwd(dy, x, gamma, ctx, ref_meta, rec)
        out = L.linear_grads(M, K, N, ln=ln)
        L.ln_linear_bwd_noalloc(dy, x, gamma, ctx, bm, rec, dx=out.dx, dw=out.dw, dbias=out.dbias,
                                dgamma=out.dgamma, dbeta=out.dbeta)
        L.sync_status()
        for name in ("dx", "dw", "dbias") + (("dgamma", "dbeta") if ln else ()):
            got, want = host(getattr(out, name)), host(getattr(ref, name))
            assert rel_fro(got, want) < TOL, (step, name)
        for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
            assert torch.equal(getattr(bm, name), getattr(ref_meta, name)), (step, name)


def test_noalloc_backward_refuses_problems_larger_than_its_scratch(L):
    M, K, N = 8192, 1024, 2048  # 16 MiB of dY codes + 16 MiB of LayerNorm gradient: too large
    a = L.CLnLinearBwd(M=M, K=K, N=N, dy=0x10000, x=0x10000, gamma=0x10000, xq=0x10000, wq=0x10000, mu=0x10000,
                       rsigma=0x10000, sinv_saved=0x10000, dx=0x10000, dw=0x10000, dbias=None, dgamma=0x10000,
                       dbeta=0x10000, dyq=None, dln=None, meta=L.CMeta(0x10000, 0x10000, 0x10000, 0x10000, 1, 16),
                       recipe=L.CRecipe(1, 16, 0, 0), defer_update=0)
    import ctypes
    st = L._c_lin_bwd_noalloc(ctypes.byref(a), None)
    assert st == L.ERR_UNSUPPORTED_SHAPE
    assert "scratch" in L.last_error()
