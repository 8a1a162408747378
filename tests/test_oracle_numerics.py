"""Pins of the oracle's LayerNorm, GELU, GEMM and bf16 rounding (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import fp8, gelu, gemm, layernorm

torch = pytest.importorskip("torch")


# ---------------------------------------------------------------- LayerNorm
def test_layernorm_pre_affine_invariants():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 96)) * rng.uniform(0.01, 30, (64, 1)) + rng.uniform(-5, 5, (64, 1))
    y, mu, rs = layernorm.forward(x, np.ones(96), np.zeros(96))
    yd = y.astype(np.float64)
    var = x.var(axis=1)
    assert np.allclose(yd.mean(axis=1), 0.0, atol=1e-5)
    # the normalised row has variance var / (var + eps), not 1
    assert np.allclose(yd.var(axis=1), var / (var + layernorm.EPS), rtol=1e-5)
    assert np.allclose(mu, x.mean(axis=1), rtol=1e-6)
    assert np.allclose(rs, 1 / np.sqrt(var + 1e-5), rtol=1e-6)


def test_layernorm_constant_row_gives_beta():
    x = np.full((3, 16), 7.25)
    g = np.linspace(0.5, 2, 16)
    b = np.linspace(-1, 1, 16)
    y, _, rs = layernorm.forward(x, g, b)
    assert np.array_equal(y, b.astype(np.float32)[None, :].repeat(3, 0))
    assert np.allclose(rs, 1 / np.sqrt(1e-5))


def test_layernorm_matches_torch_fp64():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((33, 80)) * 3 + 1
    g = 1 + 0.1 * rng.standard_normal(80)
    b = 0.1 * rng.standard_normal(80)
    y, _, _ = layernorm.forward(x, g, b)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (80,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(y, ref, rtol=2e-7, atol=2e-7)


def test_layernorm_backward_matches_autograd_and_finite_differences():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 12)) * 2
    g = 1 + 0.1 * rng.standard_normal(12)
    b = 0.1 * rng.standard_normal(12)
    dy = rng.standard_normal((5, 12))
    dx, dg, db = layernorm.backward(dy, x, g)
    xt = torch.from_numpy(x).requires_grad_()
    gt = torch.from_numpy(g).requires_grad_()
    bt = torch.from_numpy(b).requires_grad_()
    torch.nn.functional.layer_norm(xt, (12,), gt, bt, eps=1e-5).backward(torch.from_numpy(dy))
    assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-12)

    def f(xx):  # scalar objective sum(dy * LN(x)) in fp64
        xc = xx - xx.mean(axis=1, keepdims=True)
        yy = xc / np.sqrt((xc * xc).mean(axis=1, keepdims=True) + 1e-5) * g + b
        return (dy * yy).sum()
    h = 1e-6
    for i, j in itertools.product(range(5), range(0, 12, 5)):
        e = np.zeros_like(x)
        e[i, j] = h
        fd = (f(x + e) - f(x - e)) / (2 * h)
        assert abs(fd - dx[i, j]) < 1e-6 * max(1.0, abs(fd))


# ---------------------------------------------------------------- GELU
def test_gelu_fixed_points():
    assert gelu.gelu(np.array([0.0]))[0] == 0.0
    assert gelu.gelu_grad(np.array([0.0]))[0] == 0.5
    assert abs(gelu.gelu(np.array([10.0]))[0] - 10.0) < 1e-12
    assert abs(gelu.gelu(np.array([-10.0]))[0]) < 1e-12
    assert gelu.gelu_grad(np.array([0.0]), "erf")[0] == 0.5


@pytest.mark.parametrize("approx,tname", [("tanh", "tanh"), ("erf", "none")])
def test_gelu_matches_torch_and_its_derivative_matches_autograd(approx, tname):
    h = np.linspace(-8, 8, 2001)
    ht = torch.from_numpy(h).requires_grad_()
    y = torch.nn.functional.gelu(ht, approximate=tname)
    y.sum().backward()
    assert np.allclose(gelu.gelu(h, approx), y.detach().numpy(), rtol=1e-14, atol=1e-14)
    assert np.allclose(gelu.gelu_grad(h, approx), ht.grad.numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- GEMM
def _int_codes(shape, fmt, rng):
    """Codes of small integers (-4..4): exact in both formats, so every sum is exact."""
    vals = rng.integers(-4, 5, size=shape).astype(np.float32)
    return fp8.encode(vals, fmt), vals


@pytest.mark.parametrize("fa,fb", [(fp8.E4M3, fp8.E4M3), (fp8.E5M2, fp8.E4M3), (fp8.E4M3, fp8.E5M2)])
def test_gemm_equals_brute_force_on_exact_inputs(fa, fb):
    rng = np.random.default_rng(5)
    m, n, k = 7, 5, 11
    a, av = _int_codes((m, k), fa, rng)
    b, bv = _int_codes((n, k), fb, rng)
    bias = np.arange(n, dtype=np.float64) * 0.5
    c = gemm.fp8_gemm(a, fa, b, fb, 0.5, 0.25, bias)
    for i in range(m):
        for j in range(n):
            s = 0.0
            for kk in range(k):
                s += float(av[i, kk]) * float(bv[j, kk])
            assert c[i, j] == s * 0.125 + bias[j]
    assert np.array_equal(c, (av.astype(np.float64) @ bv.T.astype(np.float64)) * 0.125 + bias)


def test_gemm_dequant_factor_is_the_fp32_rounded_product():
    """The two scale_inv are multiplied in fp32 before the product is scaled (the
    state is fp32). 3 * fp32(1/3) is exactly 1 + 2^-25; in fp32 that rounds to
    1.0 (less than half an ulp away), in fp64 it stays above 1.
    A 1 x 1 GEMM of the codes of 1.0 then gives exactly 1.0 only if the factor is
    the fp32-rounded product."""
    from fractions import Fraction
    third = np.float32(1 / 3)
    exact = Fraction(3) * Fraction(float(third))
    assert exact == 1 + Fraction(1, 2 ** 25)  # below half an ulp (2^-24) of 1.0 in fp32
    one = fp8.encode(np.array([[1.0]], np.float32), fp8.E4M3)
    c = gemm.fp8_gemm(one, fp8.E4M3, one, fp8.E4M3, np.float32(3.0), third)
    assert c[0, 0] == 1.0 and float(exact) != 1.0


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(100_000) * np.exp2(rng.integers(-30, 30, 100_000)),
                        [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895e38, np.inf, -np.inf]])
    ours = gemm.to_bf16_bits(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert gemm.to_bf16_bits(np.array([np.nan]))[0] == 0x7FC0
