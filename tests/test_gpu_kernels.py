"""Parity of each CUDA kernel against the CPU oracle, through the C ABI (GPU).

Bars: FP8 codes, amaxes and the delayed-scaling state bit-exact when both sides
see the same fp32 values; LayerNorm outputs within 2e-3 relative; GEMM outputs
bit-exact on exactly representable problems and within 1e-2 relative Frobenius
otherwise.
"""
import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8 as ofp8
from oracle import fp8
from oracle import gemm as ogemm
from oracle import layernorm as oln
from oracle.delayed_scaling import ScalingState
from helpers import bf16_dev, f32_dev, host, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _scalar(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


FMT = {0: ofp8.E4M3, 1: ofp8.E5M2}


# ------------------------------------------------------------------ K2 cast
@pytest.mark.parametrize("rows,cols", [(1, 16), (300, 272), (64, 64), (129, 80), (2048, 768)])
@pytest.mark.parametrize("dt", [0, 1])
@pytest.mark.parametrize("in_fp32", [False, True])
def test_quantize_matches_oracle_bit_exact(L, rows, cols, dt, in_fp32):
    rng = np.random.default_rng(rows * 7 + cols + dt)
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-6, 6, (rows, 1)))).astype(np.float32)
    if in_fp32:
        xt = f32_dev(x)
        xv = x
    else:
        bits = synth.f32_to_bf16_bits(x)
        xt = bf16_dev(bits)
        xv = synth.bf16_bits_to_f32(bits)
    scale = np.float32(ofp8.FP8_MAX[FMT[dt]] / max(np.abs(xv).max(), 1e-30) * 0.7)
    amax = _scalar(0.0)
    out = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    out_t = torch.empty(cols, rows, dtype=torch.uint8, device="cuda")
    colsum = torch.full((cols,), 123.0, device="cuda")
    L.fp8_quantize(xt, dt, _scalar(float(scale)), amax, out=out, out_t=out_t, colsum=colsum)
    ref = ofp8.quantize(xv, scale, FMT[dt])
    assert np.array_equal(host(out), ref)
    assert np.array_equal(host(out_t), ref.T)
    assert host(amax)[0] == ofp8.amax(xv)
    cs = xv.astype(np.float64).sum(axis=0)
    assert np.allclose(host(colsum), cs, rtol=1e-4, atol=1e-4 * np.abs(xv).sum(axis=0).max())


@pytest.mark.parametrize("rows,cols,dt,with_colsum", [
    (300, 272, 0, True), (2048, 768, 1, False), (2048, 8208, 1, True),       # strip form
    (1 << 20, 16, 0, True), (45000, 384, 1, True), (32768, 544, 0, False),  # row form, 32 threads a row
    (16384, 1024, 1, True), (8192, 2048, 0, True), (4096, 4096, 1, False),  # 1-4 chunks each
    (2736, 6144, 0, True), (2048, 8192, 1, True)])                          # 64-256 threads a row
def test_quantize_bf16_rows_without_transpose_bit_exact(L, rows, cols, dt, with_colsum):
    # bf16 input and no transposed copy: tensors of 2^24 elements or more with rows of up to
    # 8192 columns take the row-streaming form (every threads-per-row / chunks-per-thread
    # shape of it here), smaller or wider ones the strip form
    rng = np.random.default_rng(rows * 5 + cols + dt)
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-6, 6, (rows, 1)))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    xv = synth.bf16_bits_to_f32(bits)
    scale = np.float32(ofp8.FP8_MAX[FMT[dt]] / max(np.abs(xv).max(), 1e-30) * 0.7)
    amax = _scalar(0.0)
    out = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    colsum = torch.full((cols,), 123.0, device="cuda") if with_colsum else None
    L.fp8_quantize(bf16_dev(bits), dt, _scalar(float(scale)), amax, out=out, colsum=colsum)
    assert np.array_equal(host(out), ofp8.quantize(xv, scale, FMT[dt]))
    assert host(amax)[0] == ofp8.amax(xv)
    if with_colsum:
        cs = xv.astype(np.float64).sum(axis=0)
        assert np.allclose(host(colsum), cs, rtol=1e-4, atol=1e-4 * np.abs(xv).sum(axis=0).max())


def test_quantize_bf16_rows_special_values(L):
    x = np.tile(np.array([[0.0, -0.0, 1e30, -1e30, np.inf, -np.inf, np.nan, 3.0] * 4], dtype=np.float32), (1 << 19, 1))
    bits = synth.f32_to_bf16_bits(x)
    amax = _scalar(5.0)
    out = torch.empty(x.shape[0], 32, dtype=torch.uint8, device="cuda")
    L.fp8_quantize(bf16_dev(bits), 0, _scalar(1.0), amax, out=out)
    got = host(out)
    ref = ofp8.quantize(synth.bf16_bits_to_f32(bits), 1.0, ofp8.E4M3)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.isnan(ofp8.decode(got[nan], ofp8.E4M3)).all()
    assert np.isnan(host(amax)[0])


def test_quantize_special_values_and_accumulating_amax(L):
    x = np.array([[0.0, -0.0, 1e30, -1e30, np.inf, -np.inf, np.nan, 3.0] * 2], dtype=np.float32)
    amax = _scalar(5.0)  # an earlier cast of the same step already saw 5
    out = torch.empty(1, 16, dtype=torch.uint8, device="cuda")
    L.fp8_quantize(f32_dev(x), 0, _scalar(1.0), amax, out=out)
    got = host(out)[0]
    ref = ofp8.quantize(x, 1.0, ofp8.E4M3)[0]
    nan = np.isnan(x[0])
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.isnan(ofp8.decode(got[nan], ofp8.E4M3)).all()
    assert np.isnan(host(amax)[0])
    amax2 = _scalar(5.0)
    L.fp8_quantize(f32_dev(np.full((3, 16), 2.0, np.float32)), 1, _scalar(1.0), amax2, out=torch.empty(3, 16, dtype=torch.uint8, device="cuda"))
    assert host(amax2)[0] == 5.0


def test_quantize_empty_rows_clears_colsum_and_keeps_amax(L):
    amax = _scalar(0.25)
    colsum = torch.full((32,), 9.0, device="cuda")
    L.fp8_quantize(torch.empty(0, 32, dtype=torch.bfloat16, device="cuda"), 0, _scalar(1.0), amax, colsum=colsum)
    torch.cuda.synchronize()
    assert host(amax)[0] == np.float32(0.25)
    assert (host(colsum) == 0).all()


# ------------------------------------------------------------------ K4 state
@pytest.mark.parametrize("Lh", [1, 2, 16, 1024])
def test_state_update_teacher_forced_bit_exact(L, Lh):
    n = 5
    dts = [0, 0, 1, 0, 1]
    rec = L.Recipe("hybrid", Lh)
    meta = L.ScalingMeta(n, Lh)
    ost = ScalingState(n, Lh)
    rng = np.random.default_rng(Lh)
    snap = torch.empty(n, device="cuda")
    for step in range(40):
        am = (np.exp(rng.standard_normal(n) * 4) * (rng.random(n) > 0.15)).astype(np.float32)
        if step == 7:
            am[1] = np.nan
        if step == 9:
            am[3] = np.inf
        if step == 11:
            am[4] = 1e-40  # subnormal amax: the scale overflows and is kept
        meta.amax_cur.copy_(torch.from_numpy(am))
        for i in range(n):
            ost.record(i, am[i])
        before = ost.scale_inv.copy()
        L.amax_history_update(meta, rec, dts, scale_inv_before=snap)
        ost.update([FMT[d] for d in dts])
        torch.cuda.synchronize()
        for name in ("scale", "scale_inv", "amax_history", "amax_cur"):
            g = host(getattr(meta, name)).astype(np.float32)
            o = getattr(ost, name)
            assert np.array_equal(g.view(np.uint32), o.view(np.uint32)), (step, name)
        assert np.array_equal(host(snap).view(np.uint32), before.view(np.uint32))


def test_meta_init(L):
    m = L.ScalingMeta(3, 7)
    torch.cuda.synchronize()
    assert (host(m.scale) == 1).all() and (host(m.scale_inv) == 1).all()
    assert (host(m.amax_history) == 0).all() and (host(m.amax_cur) == 0).all()


# ------------------------------------------------------------------ K1 / K5 LayerNorm
@pytest.mark.parametrize("M,D", [(1, 16), (300, 80), (257, 768), (64, 1280), (33, 2048), (8, 4096), (5, 8192)])
@pytest.mark.parametrize("dt", [0, 1])
def test_ln_fwd_cast(L, M, D, dt):
    x = synth.activations(M, D, dist="outliers", seed=M + D)
    g, b = synth.ln_params(D, seed=D)
    scale = np.float32(ofp8.FP8_MAX[FMT[dt]] / 12.0)
    amax = _scalar(0.0)
    ydbg = torch.empty(M, D, device="cuda")
    out, mu, rs = L.ln_fwd_cast(bf16_dev(x), bf16_dev(g), bf16_dev(b), dt, _scalar(float(scale)), amax, y_debug=ydbg)
    y_gpu = host(ydbg)
    y_ref, mu_ref, rs_ref = oln.forward(synth.bf16_bits_to_f32(x), synth.bf16_bits_to_f32(g), synth.bf16_bits_to_f32(b))
    assert rel_fro(y_gpu, y_ref) < 2e-3
    assert np.abs(y_gpu - y_ref).max() <= 2e-3 * max(1.0, np.abs(y_ref).max())
    assert np.allclose(host(mu), mu_ref, rtol=1e-4, atol=1e-5)
    assert np.allclose(host(rs), rs_ref, rtol=1e-4)
    # codes and amax: bit-exact on the kernel's own fp32 LayerNorm output
    assert np.array_equal(host(out), ofp8.quantize(y_gpu, scale, FMT[dt]))
    assert host(amax)[0] == ofp8.amax(y_gpu)


def test_ln_fwd_constant_rows_give_beta(L):
    M, D = 40, 256
    x = np.full((M, D), 0x4040, dtype=np.uint16)  # every entry 3.0
    g, b = synth.ln_params(D, seed=1)
    ydbg = torch.empty(M, D, device="cuda")
    L.ln_fwd_cast(bf16_dev(x), bf16_dev(g), bf16_dev(b), 0, _scalar(1.0), _scalar(0.0), y_debug=ydbg)
    assert np.array_equal(host(ydbg), np.broadcast_to(synth.bf16_bits_to_f32(b), (M, D)))


@pytest.mark.parametrize("M,D", [(1, 16), (300, 80), (513, 768), (100, 2048), (17, 8192)])
def test_ln_bwd(L, M, D):
    x = synth.activations(M, D, seed=M)
    g, b = synth.ln_params(D, seed=D)
    dy = synth.grad(M, D, std=0.05, seed=D)
    xt, gt = bf16_dev(x), bf16_dev(g)
    _, mu, rs = L.ln_fwd_cast(xt, gt, bf16_dev(b), 0, _scalar(1.0), _scalar(0.0))
    dx, dg, db = L.ln_bwd(bf16_dev(dy), xt, gt, mu, rs)
    rdx, rdg, rdb = oln.backward(synth.bf16_bits_to_f32(dy), synth.bf16_bits_to_f32(x), synth.bf16_bits_to_f32(g))
    assert rel_fro(host(dx), rdx) < 1e-2
    assert rel_fro(host(dg), rdg) < 1e-3
    assert rel_fro(host(db), rdb) < 1e-4


def test_ln_empty_rows(L):
    dg = torch.full((32,), 7.0, device="cuda")
    db = torch.full((32,), 7.0, device="cuda")
    e = torch.empty(0, 32, dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(32, dtype=torch.bfloat16, device="cuda")
    L.ln_bwd(e, e, gamma, torch.empty(0, device="cuda"), torch.empty(0, device="cuda"), dgamma=dg, dbeta=db)
    torch.cuda.synchronize()
    assert (host(dg) == 0).all() and (host(db) == 0).all()


# ------------------------------------------------------------------ K3 GEMM
def _int_codes(shape, fmt, rng, lo=-4, hi=4):
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return ofp8.encode(v, fmt)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 272, 400), (16, 32, 16), (520, 768, 1024)])
@pytest.mark.parametrize("adt,bdt", [(0, 0), (1, 0)])
def test_gemm_exact_integer_problems(L, a_layout, b_layout, M, N, K, adt, bdt):
    if a_layout == 1 and M % 16:
        pytest.skip("A stored [K, M] needs M % 16 == 0")
    rng = np.random.default_rng(M + N + K + 10 * a_layout + b_layout)
    a = _int_codes((M, K), FMT[adt], rng)
    b = _int_codes((N, K), FMT[bdt], rng)
    bias = synth.f32_to_bf16_bits(rng.integers(-8, 8, N).astype(np.float32))
    sa, sb = np.float32(0.5), np.float32(2.0 ** -3)
    at = torch.from_numpy(np.ascontiguousarray(a if a_layout == 0 else a.T)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(b if b_layout == 0 else b.T)).cuda()
    out = L.fp8_gemm(at, a_layout, adt, bt, b_layout, bdt, M, N, K, _scalar(float(sa)), _scalar(float(sb)), bias=bf16_dev(bias))
    ref = ogemm.fp8_gemm(a, FMT[adt], b, FMT[bdt], sa, sb, synth.bf16_bits_to_f32(bias))
    assert np.array_equal(host(out), ogemm.bf16_to_f32(ogemm.to_bf16_bits(ref)).astype(np.float64))


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(4864, 1024, 1024), (4880, 1040, 1104), (8192, 768, 256), (8208, 1152, 272)])
def test_gemm_exact_integer_problems_on_the_pair_tiles(L, a_layout, b_layout, M, N, K):
    """Enough tiles for the 256-wide CTA-pair tiles (2-SM MMA) and more K blocks
    than pipeline stages, with ragged M, N and K tails. With both operands K-major,
    N = 768 and 1152 take the 192-wide pair tiles (fewer rounds over the SMs)."""
    rng = np.random.default_rng(M + N + K + a_layout)
    a = _int_codes((M, K), fp8.E4M3, rng)
    b = _int_codes((N, K), fp8.E5M2, rng)
    at = torch.from_numpy(np.ascontiguousarray(a if a_layout == 0 else a.T)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(b if b_layout == 0 else b.T)).cuda()
    out = L.fp8_gemm(at, a_layout, 0, bt, b_layout, 1, M, N, K, _scalar(0.25), _scalar(0.5))
    ref = ogemm.fp8_gemm(a, fp8.E4M3, b, fp8.E5M2, 0.25, 0.5)
    assert np.array_equal(host(out), ogemm.bf16_to_f32(ogemm.to_bf16_bits(ref)).astype(np.float64))


@pytest.mark.parametrize("a_layout,b_layout", [(1, 1), (0, 1), (0, 0), (1, 0)])
@pytest.mark.parametrize("M,N,K", [
    (768, 3072, 8192),   # the FC2 weight gradient of the 768 -> 3072 MLP over 8192 tokens
    (520, 2832, 8208),   # ragged M (odd tile count: the pair's spare tile), N and K
    (256, 256, 8192),    # one tile
    (208, 240, 4112),    # one ragged tile, the second piece with the ragged K block
    (3072, 768, 8192),   # the FC1 weight gradient
])
def test_gemm_split_k_exact_integer_problems(L, a_layout, b_layout, M, N, K):
    """With a workspace the GEMM cuts K into pieces on separate SMs and adds the
    pieces' fp32 partials in order: integer problems stay exact, and the result
    equals the unsplit GEMM's bit for bit. The workspace's flags are left zero."""
    if a_layout == 1 and M % 16:
        pytest.skip("A stored [K, M] needs M % 16 == 0")
    nbytes = L.gemm_workspace_size(M, N, K)
    assert nbytes > 0, "this shape is meant to split"
    rng = np.random.default_rng(M + N + K + 3 * a_layout + b_layout)
    a = _int_codes((M, K), ofp8.E4M3, rng)
    b = _int_codes((N, K), ofp8.E5M2, rng)
    bias = synth.f32_to_bf16_bits(rng.integers(-8, 8, N).astype(np.float32))
    at = torch.from_numpy(np.ascontiguousarray(a if a_layout == 0 else a.T)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(b if b_layout == 0 else b.T)).cuda()
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")  # the call zeroes what it needs
    args = (at, a_layout, 0, bt, b_layout, 1, M, N, K, _scalar(0.25), _scalar(0.5))
    split = L.fp8_gemm(*args, bias=bf16_dev(bias), workspace=ws)
    whole = L.fp8_gemm(*args, bias=bf16_dev(bias))
    small = L.fp8_gemm(*args, bias=bf16_dev(bias), workspace=ws[: nbytes - 16])  # too small: runs unsplit
    L.sync_status()
    ref = ogemm.fp8_gemm(a, ofp8.E4M3, b, ofp8.E5M2, 0.25, 0.5, synth.bf16_bits_to_f32(bias))
    assert np.array_equal(host(split), ogemm.bf16_to_f32(ogemm.to_bf16_bits(ref)).astype(np.float64))
    assert torch.equal(split, whole) and torch.equal(small, whole)
    # layout: flag words, then one 128 x 256 fp32 tile per (128-row tile pair slot, 256-column tile)
    rows = -(-(-(-M // 128)) // 2) * 2
    slot_bytes = rows * (-(-N // 256)) * 128 * 256 * 4
    flag_bytes = nbytes - slot_bytes
    w = ws.cpu().numpy()
    assert 0 < flag_bytes and flag_bytes % 256 == 0
    assert not w[:flag_bytes].any(), "the flags are left zero"
    assert (w[flag_bytes:] != 0xAB).mean() > 0.5, "the exchanged partials went to the slots"


def test_gemm_split_k_random_codes_within_tolerance(L):
    M, N, K = 768, 3072, 8192
    rng = np.random.default_rng(7)
    a = ofp8.encode(rng.standard_normal((M, K)).astype(np.float32) * 30, ofp8.E5M2)
    b = ofp8.encode(rng.standard_normal((N, K)).astype(np.float32) * 40, ofp8.E4M3)
    sa, sb = np.float32(1 / 30.0), np.float32(1 / 40.0)
    at = torch.from_numpy(np.ascontiguousarray(a.T)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(b.T)).cuda()
    ws = torch.zeros(L.gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    out = L.fp8_gemm(at, 1, 1, bt, 1, 0, M, N, K, _scalar(float(sa)), _scalar(float(sb)), workspace=ws)
    L.sync_status()
    ref = ogemm.fp8_gemm(a, ofp8.E5M2, b, ofp8.E4M3, sa, sb)
    got = host(out)
    assert rel_fro(got, ref) < 1e-2
    assert np.abs(got - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 1)])
def test_gemm_random_codes_within_tolerance(L, a_layout, b_layout):
    M, N, K = 384, 512, 3072
    rng = np.random.default_rng(42)
    a = ofp8.encode(rng.standard_normal((M, K)).astype(np.float32) * 30, ofp8.E4M3)
    b = ofp8.encode(rng.standard_normal((N, K)).astype(np.float32) * 2000, ofp8.E5M2)
    sa, sb = np.float32(1 / 30.0), np.float32(1 / 2000.0)
    at = torch.from_numpy(np.ascontiguousarray(a if a_layout == 0 else a.T)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(b if b_layout == 0 else b.T)).cuda()
    out = L.fp8_gemm(at, a_layout, 0, bt, b_layout, 1, M, N, K, _scalar(float(sa)), _scalar(float(sb)))
    ref = ogemm.fp8_gemm(a, ofp8.E4M3, b, ofp8.E5M2, sa, sb)
    got = host(out)
    assert rel_fro(got, ref) < 1e-2
    assert np.abs(got - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


# ------------------------------------------------------------------ failure path
def test_bounded_wait_reports_timeout_and_context_survives(L):
    L.sync_status()  # clear anything earlier
    L.lnfp8_selftest_timeout(2_000_000)  # 2 ms
    with pytest.raises(L.LnFp8Error) as e:
        L.sync_status()
    assert e.value.status == L.ERR_TIMEOUT
    L.sync_status()  # cleared
    t = torch.ones(1024, device="cuda")
    assert float(t.sum()) == 1024.0
