"""ln_linear_bwd_noalloc: the LayerNormLinear backward for callers that cannot
allocate device memory (GPU).

Some callers may not call cudaMalloc: a plug-in that a host framework hands
only the tensors of one layer, or a runtime whose device memory is fixed before
start-up. Such a caller passes inputs and outputs only; the dY codes and the
LayerNorm-output gradient live in the library's own fixed scratch array. The
tests check, through the C ABI:
  * two calls in a row give the same results as ln_linear_bwd with
    caller-provided scratch, within the tolerance the other parity tests use,
    and the same delayed-scaling state bit for bit;
  * the call takes no device memory: the GPU's free memory is the same
    before and after the second call;
  * a problem larger than the scratch is refused before anything is enqueued
    (real buffers of the declared sizes, whose contents stay untouched).

The file is named so that pytest collects it last: if it fails, a run that
stops at the first failure (-x) has already run every other test. It passes
both alone in a fresh process and after the other tests (its first call on the
device does the one-time address lookup either way).
"""
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


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


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
        free0 = _free_bytes()
        L.ln_linear_bwd_noalloc(dy, x, gamma, ctx, bm, rec, dx=out.dx, dw=out.dw, dbias=out.dbias,
                                dgamma=out.dgamma, dbeta=out.dbeta)
        L.sync_status()
        free1 = _free_bytes()
        if step == 1:  # the first call may load the kernels' code; the second reuses everything
            assert free1 == free0, f"device memory changed by {free0 - free1} bytes"
        for name in ("dx", "dw", "dbias") + (("dgamma", "dbeta") if ln else ()):
            got, want = host(getattr(out, name)), host(getattr(ref, name))
            assert rel_fro(got, want) < TOL, (step, name)
        for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
            assert torch.equal(getattr(bm, name), getattr(ref_meta, name)), (step, name)


def test_noalloc_backward_refuses_problems_larger_than_its_scratch(L):
    # 9 MiB of dY codes + 8 MiB of LayerNorm-output gradient: one MiB over the 16 MiB scratch
    M, K, N = 4096, 1024, 2304
    rec = L.Recipe("hybrid", 16)
    dev = "cuda"
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    dy = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)
    gamma = torch.ones(K, dtype=torch.bfloat16, device=dev)
    ctx = L.linear_ctx(M, K, N, ln=True, device=dev)
    for t in (ctx.xq, ctx.wq, ctx.mu, ctx.rsigma, ctx.sinv_saved):
        t.zero_()
    bm = L.ScalingMeta(1, 16)
    sentinel = 0x3F80  # bf16 1.0
    dx = torch.full((M, K), 1.0, dtype=torch.bfloat16, device=dev)
    dw = torch.full((N, K), 1.0, dtype=torch.bfloat16, device=dev)
    dbias = torch.full((N,), 7.0, device=dev)
    dgamma = torch.full((K,), 7.0, device=dev)
    dbeta = torch.full((K,), 7.0, device=dev)
    state0 = {k: v.clone() for k, v in bm.state_dict().items()}
    torch.cuda.synchronize()
    with pytest.raises(L.LnFp8Error) as e:
        L.ln_linear_bwd_noalloc(dy, x, gamma, ctx, bm, rec, dx=dx, dw=dw, dbias=dbias, dgamma=dgamma, dbeta=dbeta)
    assert e.value.status == L.ERR_UNSUPPORTED_SHAPE
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    # refused before anything was enqueued: outputs and state untouched
    assert (dx.view(torch.int16) == sentinel).all() and (dw.view(torch.int16) == sentinel).all()
    assert (dbias == 7.0).all() and (dgamma == 7.0).all() and (dbeta == 7.0).all()
    for k, v in bm.state_dict().items():
        assert torch.equal(v, state0[k]), k
