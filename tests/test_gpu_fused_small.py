"""The one-launch LayerNormLinear / Linear forward for few tokens (GPU).

The fused path computes, per 128 x 128 output tile, the LayerNorm + amax + cast
of its token rows straight into the tensor cores' A operand in shared memory
and the weight cast into the B operand, then the GEMM, dequantisation and bias;
the state update follows as a launch of its own. Each of its steps is the
separate kernels' own arithmetic in the same order, so everything it writes
must equal the separate launches' results bit for bit: the output, the saved
codes, mu and rsigma, the LayerNorm debug dump, the saved scale_inv and the
state after the update, over several steps (the later ones cast with scales
from the earlier ones). Parity of both paths with the oracle is in
tests/test_gpu_modules.py (run_linear, path 1 and 2).
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from helpers import bf16_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _same_state(a, b):
    return all(torch.equal(getattr(a, k), getattr(b, k)) for k in ("scale", "scale_inv", "amax_history", "amax_cur"))


@pytest.mark.parametrize("M,K,N", [(256, 768, 2304), (1, 16, 16), (100, 192, 400), (300, 768, 2304),
                                   (256, 640, 1040), (129, 400, 272), (513, 16, 144)])
@pytest.mark.parametrize("ln", [True, False])
@pytest.mark.parametrize("fmt", ["e4m3", "hybrid", "e5m2"])
def test_fused_forward_equals_separate_launches(L, M, K, N, ln, fmt):
    rec = L.Recipe(fmt, 4)
    p = synth.linear_params(N, K, ln=ln, bias_std=0.02, seed=M + K + N)
    w, b = bf16_dev(p["w"]), bf16_dev(p["b"])
    g = bf16_dev(p["gamma"]) if ln else None
    be = bf16_dev(p["beta"]) if ln else None
    metas = [L.ScalingMeta(2, 4), L.ScalingMeta(2, 4)]
    for step in range(3):
        x = bf16_dev(synth.activations(M, K, dist="outliers", seed=K, step=step))
        outs = []
        for meta, path in zip(metas, (L.PATH_FUSED, L.PATH_SEPARATE)):
            y, ctx = L.ln_linear_fwd(x, g, be, w, b, meta, rec, debug=ln, path=path)
            outs.append((y, ctx))
        L.sync_status()
        (y0, c0), (y1, c1) = outs
        assert torch.equal(y0, y1), (step, "y")
        for name in ("xq", "wq", "sinv_saved") + (("mu", "rsigma", "ln_out_debug") if ln else ()):
            assert torch.equal(getattr(c0, name), getattr(c1, name)), (step, name)
        assert _same_state(metas[0], metas[1]), step


def test_fused_forward_with_fp8_stored_weight(L):
    M, K, N = 256, 768, 2304
    rec = L.Recipe("hybrid", 16)
    p = synth.linear_params(N, K, bias_std=0.02, seed=5)
    wt = bf16_dev(p["w"])
    fw = L.quantize_weight(wt, rec)
    metas = [L.ScalingMeta(2, 16), L.ScalingMeta(2, 16)]
    for step in range(2):
        x = bf16_dev(synth.activations(M, K, seed=5, step=step))
        outs = [L.ln_linear_fwd(x, bf16_dev(p["gamma"]), bf16_dev(p["beta"]), fw, bf16_dev(p["b"]), m, rec, path=path)
                for m, path in zip(metas, (L.PATH_FUSED, L.PATH_SEPARATE))]
        L.sync_status()
        assert torch.equal(outs[0][0], outs[1][0])
        assert torch.equal(outs[0][1].xq, outs[1][1].xq) and torch.equal(outs[0][1].sinv_saved, outs[1][1].sinv_saved)
        assert _same_state(metas[0], metas[1])


def test_fused_path_in_a_cuda_graph_and_its_limits(L):
    M, K, N = 64, 768, 512
    rec = L.Recipe("e4m3", 16)
    p = synth.linear_params(N, K, seed=9)
    args = [bf16_dev(p[k]) for k in ("gamma", "beta", "w", "b")]
    x = bf16_dev(synth.activations(M, K, seed=9))
    m0, m1 = L.ScalingMeta(2, 16), L.ScalingMeta(2, 16)
    y0, _ = L.ln_linear_fwd(x, args[0], args[1], args[2], args[3], m0, rec, path=L.PATH_FUSED)
    ctx = L.linear_ctx(M, K, N)
    y1 = torch.empty_like(y0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        L.ln_linear_fwd(x, args[0], args[1], args[2], args[3], m1, rec, y=y1, ctx=ctx, path=L.PATH_FUSED)
    gr.replay()
    torch.cuda.synchronize()
    L.sync_status()
    assert torch.equal(y0, y1) and _same_state(m0, m1)
    # K above the shared-memory panels, and a fused residual add, are refused on the fused path
    big = bf16_dev(synth.activations(8, 1024, seed=1))
    wb = bf16_dev(synth.weight(16, 1024))
    gb = torch.ones(1024, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.LnFp8Error) as e:
        L.ln_linear_fwd(big, gb, gb, wb, None, L.ScalingMeta(2, 16), rec, path=L.PATH_FUSED)
    assert e.value.status == L.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(L.LnFp8Error) as e:
        L.ln_linear_fwd(x, args[0], args[1], args[2], args[3], L.ScalingMeta(2, 16), rec, residual=x,
                        path=L.PATH_FUSED)
    assert e.value.status == L.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(L.LnFp8Error) as e:
        L.ln_linear_fwd(x, args[0], args[1], args[2], args[3], L.ScalingMeta(2, 16), rec, path=7)
    assert e.value.status == L.ERR_INVALID_ARG
