"""Worker functions for the process pool of the full-size parity tests.

The pool is started with the spawn method: the parent process holds a CUDA
context, which a forked child would inherit. Each worker runs the seeded input
generator or the oracle's scaled FP8 cast on one slice of a large tensor. The
cast is elementwise, so casting the row slices separately gives the same codes
as one call over the whole tensor. No arithmetic of the method lives here.
"""
import numpy as np

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8


def quantize_bf16_rows(args):
    """oracle cast of a slice of a bf16 tensor (bits) with one fp32 scale."""
    bits, scale, fmt = args
    return fp8.quantize(synth.bf16_bits_to_f32(bits), np.float32(scale), fmt)


def pquantize(pool, bits, scale, fmt, parts=16):
    """The oracle's cast of a whole bf16 tensor, its rows split over the pool."""
    chunks = np.array_split(np.ascontiguousarray(bits), min(parts, max(1, bits.shape[0])), axis=0)
    return np.concatenate(pool.map(quantize_bf16_rows, [(c, np.float32(scale), fmt) for c in chunks]), axis=0)


def stack_layer_params(args):
    """Seeded parameters of one layer of the block stack (names as the benchmark's stack)."""
    layer, d, f, seed, bias_std = args
    qkv = synth.linear_params(3 * d, d, seed=seed, layer=layer, bias_std=bias_std, wtid=synth.TID["wqkv"],
                              btid=synth.TID["bqkv"])
    proj = synth.linear_params(d, d, seed=seed, layer=layer, ln=False, bias_std=bias_std,
                               wtid=synth.TID["wproj"], btid=synth.TID["bproj"])
    mlp = synth.mlp_params(d, f, seed=seed, layer=layer, bias_std=bias_std)
    return dict(wqkv=qkv["w"], bqkv=qkv["b"], g1=qkv["gamma"], be1=qkv["beta"], wproj=proj["w"], bproj=proj["b"],
                g2=mlp["gamma"], be2=mlp["beta"], w1=mlp["w1"], b1=mlp["b1"], w2=mlp["w2"], b2=mlp["b2"])


def draw(args):
    """One whole seeded input tensor, (kind, rows, cols, keywords) -> bf16 bits; kind
    "act" is synth.activations, anything else synth.grad. (Each tensor is one draw of
    its generator, so tensors, not row slices, are spread over the workers.)"""
    kind, rows, cols, kw = args
    if kind == "act":
        return synth.activations(rows, cols, **kw)
    return synth.grad(rows, cols, **kw)


def mlp_column_run(args):
    """The oracle LayerNormMLP step over all tokens, restricted to the FFN columns
    `cols` (W1 rows, b1 entries and W2 columns given as the oracle's codes of those
    slices); returns the column-wise results the GPU tests compare."""
    from oracle import modules as omod
    x, dy, p, cols, w1q_c, w2q_c, fpre, bpre, rec = args
    si = fpre.scale_inv
    _, cc, ac = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], None, p["b1"][cols], None, p["b2"], fpre.copy(), rec,
                                fp8_weights=((w1q_c, si[1]), (w2q_c, si[3])))
    gc = omod.ln_mlp_bwd(dy, cc, bpre.copy(), rec)
    return dict(h=ac["h"], a=ac["a"], y=ac["y"], aq=cc.aq, dh=gc["dh"], dhq=gc["dhq"], db1=gc["db1"],
                dw1=gc["dw1"], dw2=gc["dw2"], db2=gc["db2"], dyq=gc["dyq"])
