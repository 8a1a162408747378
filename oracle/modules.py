"""LayerNormLinear / Linear and LayerNormMLP, forward and backward, under FP8
delayed scaling (oracle; test infrastructure only).

The modules are ``te.LayerNormLinear(H, 3*H)``, ``te.Linear(H, H, bias=True)``
and ``te.LayerNormMLP(H, 4*H)`` run inside ``te.fp8_autocast`` with the
delayed-scaling recipe (TE tutorial, code blocks 1 and 3; Turbo-charging guide,
"The building blocks: fused modules you'll use" and "Playing with
lower-precision formats: BF16 vs FP8": activations are converted to FP8 with
their tracked scale and gradients come back in BF16/FP32 for the optimizer).
The pages show only the Python surface, so the dataflow below is the plain
reading of that surface, step by step:

LayerNormMLP forward (fwd state slots: 0 LN output, 1 W1, 2 GELU output A, 3 W2)
  y, mu, rsigma = LayerNorm(X)                    fp32 y
  yq  = cast(y,  scale[0]);  amax[0] <- max|y|
  W1q = cast(W1, scale[1]);  amax[1] <- max|W1|
  W2q = cast(W2, scale[3]);  amax[3] <- max|W2|
  H   = bf16( (yq . W1q^T) * (sinv[0]*sinv[1]) + b1 )
  A   = gelu(H)  (fp32, from the bf16 H)
  Aq  = cast(A,  scale[2]);  amax[2] <- max|A|
  Y   = bf16( (Aq . W2q^T) * (sinv[2]*sinv[3]) + b2 )
  then the end-of-step update of the forward state.
LayerNormMLP backward (bwd state slots: 0 dY, 1 dH); sinv_f are the forward's
scale_inv as they were when the forward cast its tensors:
  dYq = cast(dY, gscale[0]); amax <- max|dY|;  db2 = sum_rows dY
  dA  = (dYq . W2q) * (gsinv[0]*sinv_f[3])          fp32 inside the fused epilogue
  dH  = dA * gelu'(H)                                fp32
  dHq = cast(dH, gscale[1]); amax <- max|dH|;  db1 = sum_rows dH
  dW2 = bf16( (dYq^T . Aq) * (gsinv[0]*sinv_f[2]) )
  dLN = bf16( (dHq . W1q) * (gsinv[1]*sinv_f[1]) )
  dW1 = bf16( (dHq^T . yq) * (gsinv[1]*sinv_f[0]) )
  dX, dgamma, dbeta = LayerNorm backward of dLN; then the backward state update.
Readings (the pages are silent): GELU is applied to the bf16 H that is saved
for the backward; dA and dH stay fp32 between the dgrad GEMM and the E5M2 cast;
bias and LayerNorm gradients are returned in fp32, dX and weight gradients in
bf16.

LayerNormLinear (fwd slots 0 input, 1 W; bwd slot 0 dY) is the same with one
GEMM; with no LayerNorm (gamma None) it is te.Linear and X itself is cast.

``exact=True`` switches every cast and every intermediate rounding off (fp64
throughout), which reduces these functions to the textbook fp64 LayerNorm / MLP
and their autograd gradients: that is how the composition is pinned. With
quantisation on, the end-to-end values have no pin beyond their components
(parity unpinned beyond the component pins).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import fp8 as _fp8
from . import gelu as _gelu
from . import layernorm as _ln
from .delayed_scaling import Recipe, ScalingState
from .gemm import bf16_to_f32, dequant_scale, to_bf16_bits


class _Numerics:
    def __init__(self, exact: bool):
        self.exact = exact

    def f32(self, x):
        return np.asarray(x, np.float64) if self.exact else np.asarray(x, np.float64).astype(np.float32)

    def cast(self, x, scale, fmt):
        if self.exact:
            return np.asarray(x, np.float64)
        return _fp8.quantize(x, scale, fmt)

    def dec(self, payload, fmt):
        if self.exact:
            return payload
        return _fp8.decode(payload, fmt)

    def amax(self, x):
        return np.float32(0) if self.exact else _fp8.amax(x)

    def bf16(self, x):
        if self.exact:
            return np.asarray(x, np.float64)
        return bf16_to_f32(to_bf16_bits(x)).astype(np.float64)

    def dq(self, sinv_a, sinv_b):
        return 1.0 if self.exact else np.float64(dequant_scale(sinv_a, sinv_b))


def _in(bits_or_vals):
    """Module inputs arrive as bf16 bit patterns (uint16) or as float values."""
    a = np.asarray(bits_or_vals)
    if a.dtype == np.uint16:
        return bf16_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


@dataclass
class Ctx:
    """Tensors saved by a forward for its backward."""
    x: np.ndarray
    gamma: np.ndarray | None
    yq: np.ndarray
    wq: list
    sinv: np.ndarray
    h: np.ndarray | None = None
    aq: np.ndarray | None = None
    fmt: str = _fp8.E4M3
    debug: dict = field(default_factory=dict)


def quantize_weight(w, recipe: Recipe, state: ScalingState | None = None):
    """A weight converted once to FP8 storage (TE tutorial, closing list of
    things to try: ``fp8_model_init()`` keeps the weights themselves in FP8 for
    inference). The pages name the feature only; the reading here is the
    delayed-scaling rule applied to the weight's own state (n = 1, fresh unless
    given): record max|W|, run the end-of-step update (so with a fresh state
    scale = fp8_max / max|W| / 2^margin), cast W with that scale, and record the
    cast's amax as every cast does. Returns (codes, scale_inv, state)."""
    fmt = recipe.fwd_fmt()
    st = state if state is not None else ScalingState(1, 1)
    W = _in(w)
    st.record(0, _fp8.amax(W.astype(np.float32)))
    st.update([fmt], recipe.amax_compute_algo, recipe.margin)
    codes = _fp8.quantize(W, st.scale[0], fmt)
    st.record(0, _fp8.amax(W.astype(np.float32)))
    return codes, np.float32(st.scale_inv[0]), st


def _residual_sum(X, residual, nm):
    """The residual connection ahead of a block's LayerNorm (TE tutorial code
    block 2, the plain-PyTorch block: x = x + a; x + mlp(ln2(x))): the module's
    input is the bf16 sum of the two bf16 tensors."""
    return nm.bf16(X + _in(residual))


def ln_linear_fwd(x, gamma, beta, w, b, state: ScalingState, recipe: Recipe, *,
                  exact: bool = False, update: bool = True, fp8_weight=None, residual=None):
    """LayerNormLinear (gamma given) or Linear (gamma None) forward.

    fp8_weight: None, or (codes, scale_inv) of a weight kept in FP8 (see
    quantize_weight); then w is unused, no weight is cast, slot 1 records no
    amax, and the GEMM and the saved scale_inv take the weight's own value.
    Returns (Y [M, N] float values rounded to bf16, ctx, aux) where aux holds
    mu, rsigma and the fp32 pre-cast LN output."""
    nm = _Numerics(exact)
    fmt = recipe.fwd_fmt()
    if fp8_weight is not None and exact:
        raise ValueError("exact=True has no FP8-stored weight")
    X = _in(x)
    aux = {}
    if residual is not None:
        if gamma is None:
            raise ValueError("the residual add precedes a LayerNorm")
        X = _residual_sum(X, residual, nm)
        aux["x_sum"] = X
    if gamma is not None:
        y, mu, rs = _ln.forward(X, _in(gamma), _in(beta))
        if exact:
            xc = X - X.mean(axis=1, keepdims=True)
            y = xc / np.sqrt((xc * xc).mean(axis=1, keepdims=True) + _ln.EPS) * _in(gamma) + _in(beta)
        aux.update(mu=mu, rsigma=rs)
    else:
        y = X
    y = nm.f32(y)
    aux["y"] = y
    state.record(0, nm.amax(y))
    yq = nm.cast(y, state.scale[0], fmt)
    sinv = state.scale_inv.copy()
    if fp8_weight is None:
        W = _in(w)
        state.record(1, nm.amax(W.astype(np.float32)))
        wq = nm.cast(W, state.scale[1], fmt)
    else:
        wq, sinv[1] = fp8_weight
    acc = nm.dec(yq, fmt) @ nm.dec(wq, fmt).T
    out = acc * nm.dq(sinv[0], sinv[1])
    if b is not None:
        out = out + _in(b)[None, :]
    Y = nm.bf16(out)
    if update:
        state.update([fmt, fmt], recipe.amax_compute_algo, recipe.margin)
    ctx = Ctx(x=X, gamma=None if gamma is None else _in(gamma), yq=yq, wq=[wq], sinv=sinv, fmt=fmt)
    return Y, ctx, aux


def ln_linear_bwd(dy, ctx: Ctx, gstate: ScalingState, recipe: Recipe, *,
                  exact: bool = False, update: bool = True):
    """Backward of ln_linear_fwd: returns dict(dx, dw, db, dgamma, dbeta, dyq)."""
    nm = _Numerics(exact)
    gfmt = recipe.bwd_fmt()
    fmt = ctx.fmt
    dY = _in(dy)
    gstate.record(0, nm.amax(dY.astype(np.float32)))
    dyq = nm.cast(dY, gstate.scale[0], gfmt)
    gsinv = gstate.scale_inv.copy()
    db = dY.sum(axis=0)
    dyv = nm.dec(dyq, gfmt)
    dln = nm.bf16(dyv @ nm.dec(ctx.wq[0], fmt) * nm.dq(gsinv[0], ctx.sinv[1]))
    dw = nm.bf16(dyv.T @ nm.dec(ctx.yq, fmt) * nm.dq(gsinv[0], ctx.sinv[0]))
    res = dict(dw=dw, db=db, dyq=dyq)
    if ctx.gamma is not None:
        dx, dg, dbeta = _ln.backward(dln, ctx.x, ctx.gamma)
        res.update(dx=nm.bf16(dx), dgamma=dg, dbeta=dbeta, dln=dln)
    else:
        res.update(dx=dln, dgamma=None, dbeta=None, dln=dln)
    if update:
        gstate.update([gfmt], recipe.amax_compute_algo, recipe.margin)
    return res


def ln_mlp_fwd(x, gamma, beta, w1, b1, w2, b2, state: ScalingState, recipe: Recipe, *,
               exact: bool = False, update: bool = True, gelu_approx: str = "tanh", fp8_weights=None,
               residual=None):
    """LayerNormMLP forward. Returns (Y, ctx, aux); aux holds mu, rsigma, the
    fp32 pre-cast LN output y and GELU output a, and the bf16 H.

    fp8_weights: None, or ((W1 codes, scale_inv), (W2 codes, scale_inv)) of
    weights kept in FP8 (see quantize_weight); then w1 and w2 are unused, slots
    1 and 3 record no amax, and their scale_inv come from the weights."""
    nm = _Numerics(exact)
    fmt = recipe.fwd_fmt()
    if fp8_weights is not None and exact:
        raise ValueError("exact=True has no FP8-stored weights")
    X = _in(x)
    if residual is not None:
        X = _residual_sum(X, residual, nm)
    G = _in(gamma)
    y, mu, rs = _ln.forward(X, G, _in(beta))
    if exact:
        xc = X - X.mean(axis=1, keepdims=True)
        y = xc / np.sqrt((xc * xc).mean(axis=1, keepdims=True) + _ln.EPS) * G + _in(beta)
    y = nm.f32(y)
    state.record(0, nm.amax(y))
    yq = nm.cast(y, state.scale[0], fmt)
    sinv = state.scale_inv.copy()
    if fp8_weights is None:
        W1, W2 = _in(w1), _in(w2)
        state.record(1, nm.amax(W1.astype(np.float32)))
        w1q = nm.cast(W1, state.scale[1], fmt)
        state.record(3, nm.amax(W2.astype(np.float32)))
        w2q = nm.cast(W2, state.scale[3], fmt)
    else:
        (w1q, sinv[1]), (w2q, sinv[3]) = fp8_weights
    h = nm.dec(yq, fmt) @ nm.dec(w1q, fmt).T * nm.dq(sinv[0], sinv[1])
    if b1 is not None:
        h = h + _in(b1)[None, :]
    H = nm.bf16(h)
    a = nm.f32(_gelu.gelu(H, gelu_approx))
    state.record(2, nm.amax(a))
    aq = nm.cast(a, state.scale[2], fmt)
    out = nm.dec(aq, fmt) @ nm.dec(w2q, fmt).T * nm.dq(sinv[2], sinv[3])
    if b2 is not None:
        out = out + _in(b2)[None, :]
    Y = nm.bf16(out)
    if update:
        state.update([fmt] * 4, recipe.amax_compute_algo, recipe.margin)
    ctx = Ctx(x=X, gamma=G, yq=yq, wq=[w1q, w2q], sinv=sinv, h=H, aq=aq, fmt=fmt)
    aux = dict(mu=mu, rsigma=rs, y=y, a=a, h=H)
    if residual is not None:
        aux["x_sum"] = X
    return Y, ctx, aux


def ln_mlp_bwd(dy, ctx: Ctx, gstate: ScalingState, recipe: Recipe, *,
               exact: bool = False, update: bool = True, gelu_approx: str = "tanh"):
    """LayerNormMLP backward. Returns dict(dx, dgamma, dbeta, dw1, db1, dw2,
    db2) plus the intermediate dyq, dh (fp32 pre-cast), dhq and dln."""
    nm = _Numerics(exact)
    gfmt = recipe.bwd_fmt()
    fmt = ctx.fmt
    dY = _in(dy)
    gstate.record(0, nm.amax(dY.astype(np.float32)))
    dyq = nm.cast(dY, gstate.scale[0], gfmt)
    db2 = dY.sum(axis=0)
    gsinv0 = gstate.scale_inv[0]
    w1q, w2q = ctx.wq
    dyv = nm.dec(dyq, gfmt)
    da = dyv @ nm.dec(w2q, fmt) * nm.dq(gsinv0, ctx.sinv[3])
    dh = nm.f32(da * _gelu.gelu_grad(ctx.h, gelu_approx))
    gstate.record(1, nm.amax(dh))
    dhq = nm.cast(dh, gstate.scale[1], gfmt)
    gsinv1 = gstate.scale_inv[1]
    db1 = np.asarray(dh, np.float64).sum(axis=0)
    dw2 = nm.bf16(dyv.T @ nm.dec(ctx.aq, fmt) * nm.dq(gsinv0, ctx.sinv[2]))
    dhv = nm.dec(dhq, gfmt)
    dln = nm.bf16(dhv @ nm.dec(w1q, fmt) * nm.dq(gsinv1, ctx.sinv[1]))
    dw1 = nm.bf16(dhv.T @ nm.dec(ctx.yq, fmt) * nm.dq(gsinv1, ctx.sinv[0]))
    dx, dg, dbeta = _ln.backward(dln, ctx.x, ctx.gamma)
    if update:
        gstate.update([gfmt, gfmt], recipe.amax_compute_algo, recipe.margin)
    return dict(dx=nm.bf16(dx), dgamma=dg, dbeta=dbeta, dw1=dw1, db1=db1, dw2=dw2, db2=db2,
                dyq=dyq, dh=dh, dhq=dhq, dln=dln)
