"""Python binding of liblnfp8 (the C ABI declared in include/lnfp8.h).

Argument marshalling only: PyTorch provides device memory and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels. If
the shared library has not been built, importing this module raises.

Names follow the C ABI: lnfp8_meta_init, amax_history_update, fp8_quantize,
ln_fwd_cast, ln_bwd, fp8_gemm, ln_linear_fwd / ln_linear_bwd,
ln_mlp_fwd / ln_mlp_bwd.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblnfp8.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"liblnfp8.so is not built ({LIB_PATH}); run fp8_delayed_scaling_row_gb300.build.build_library()")
_lib = C.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(6)
E4M3, E5M2 = 0, 1
FORMAT_E4M3, FORMAT_HYBRID, FORMAT_E5M2 = 0, 1, 2
_FORMATS = {"e4m3": FORMAT_E4M3, "hybrid": FORMAT_HYBRID, "e5m2": FORMAT_E5M2}

EXPORTED = [
    "lnfp8_last_error", "lnfp8_sync_status", "lnfp8_version", "lnfp8_selftest_timeout", "lnfp8_launch_count",
    "lnfp8_profile_enable", "lnfp8_profile_sample", "lnfp8_profile_collect", "lnfp8_profile_get", "lnfp8_meta_init", "amax_history_update", "amax_history_update_many",
    "fp8_quantize", "fp8_weight_quantize", "ln_fwd_cast", "ln_bwd", "fp8_gemm", "ln_linear_fwd", "ln_linear_bwd",
    "ln_linear_bwd_noalloc", "ln_mlp_fwd", "ln_mlp_bwd", "lnfp8_gemm_workspace_size",
    "lnfp8_ln_linear_bwd_workspace_size", "lnfp8_ln_mlp_bwd_workspace_size", "lnfp8_ln_mlp_fwd_workspace_size",
    "lnfp8_ctx_bytes", "lnfp8_ctx_offsets",
]
OP_LN_LINEAR, OP_LINEAR, OP_LN_MLP = 0, 1, 2


class LnFp8Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lnfp8 status {status}: {msg}")
        self.status = status


# ------------------------------------------------------------------ C structs
class CRecipe(C.Structure):
    _fields_ = [("format", C.c_int), ("history_len", C.c_int), ("algo", C.c_int), ("margin", C.c_int)]


class CMeta(C.Structure):
    _fields_ = [("scale", C.c_void_p), ("scale_inv", C.c_void_p), ("amax_history", C.c_void_p),
                ("amax_cur", C.c_void_p), ("n", C.c_int), ("history_len", C.c_int)]


_P = C.c_void_p
_I64 = C.c_int64


class CLnLinearFwd(C.Structure):
    _fields_ = [("M", _I64), ("K", _I64), ("N", _I64), ("x", _P), ("gamma", _P), ("beta", _P), ("eps", C.c_float),
                ("w", _P), ("bias", _P), ("y", _P), ("xq", _P), ("wq", _P), ("mu", _P), ("rsigma", _P),
                ("sinv_saved", _P), ("meta", CMeta), ("recipe", CRecipe), ("defer_update", C.c_int),
                ("ln_out_debug", _P), ("w_scale_inv", _P), ("residual", _P), ("x_sum", _P), ("path", C.c_int)]


PATH_AUTO, PATH_FUSED, PATH_SEPARATE = 0, 1, 2


class CLnLinearBwd(C.Structure):
    _fields_ = [("M", _I64), ("K", _I64), ("N", _I64), ("dy", _P), ("x", _P), ("gamma", _P), ("xq", _P),
                ("wq", _P), ("mu", _P), ("rsigma", _P), ("sinv_saved", _P), ("dx", _P), ("dw", _P), ("dbias", _P),
                ("dgamma", _P), ("dbeta", _P), ("dyq", _P), ("dln", _P), ("meta", CMeta), ("recipe", CRecipe),
                ("defer_update", C.c_int), ("gemm_ws", _P), ("gemm_ws_bytes", _I64)]


class CLnMlpFwd(C.Structure):
    _fields_ = [("M", _I64), ("D", _I64), ("F", _I64), ("x", _P), ("gamma", _P), ("beta", _P), ("eps", C.c_float),
                ("w1", _P), ("b1", _P), ("w2", _P), ("b2", _P), ("y", _P), ("lnq", _P), ("mu", _P), ("rsigma", _P),
                ("w1q", _P), ("w2q", _P), ("h", _P), ("aq", _P), ("sinv_saved", _P), ("meta", CMeta),
                ("recipe", CRecipe), ("defer_update", C.c_int), ("ln_out_debug", _P), ("act_debug", _P),
                ("gemm_ws", _P), ("gemm_ws_bytes", _I64), ("w1_scale_inv", _P), ("w2_scale_inv", _P),
                ("residual", _P), ("x_sum", _P)]


class CLnMlpBwd(C.Structure):
    _fields_ = [("M", _I64), ("D", _I64), ("F", _I64), ("dy", _P), ("x", _P), ("gamma", _P), ("lnq", _P),
                ("mu", _P), ("rsigma", _P), ("w1q", _P), ("w2q", _P), ("h", _P), ("aq", _P), ("sinv_saved", _P),
                ("dx", _P), ("dgamma", _P), ("dbeta", _P), ("dw1", _P), ("db1", _P), ("dw2", _P), ("db2", _P),
                ("dyq", _P), ("dhq", _P), ("dln", _P), ("meta", CMeta), ("recipe", CRecipe),
                ("defer_update", C.c_int), ("dh_debug", _P), ("gemm_ws", _P), ("gemm_ws_bytes", _I64)]


def _sig(name, args, res=C.c_int):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_lib.lnfp8_last_error.restype = C.c_char_p
_lib.lnfp8_last_error.argtypes = []
_c_sync = _sig("lnfp8_sync_status", [_P])
_c_version = _sig("lnfp8_version", [])
_c_selftest = _sig("lnfp8_selftest_timeout", [_I64, _P])
_c_launch_count = _sig("lnfp8_launch_count", [], C.c_longlong)
_c_prof_enable = _sig("lnfp8_profile_enable", [C.c_int])
_c_prof_sample = _sig("lnfp8_profile_sample", [])
_c_prof_collect = _sig("lnfp8_profile_collect", [])
_c_prof_get = _sig("lnfp8_profile_get", [C.c_int, C.POINTER(C.c_char_p), C.POINTER(C.c_double),
                                         C.POINTER(C.c_longlong)])
_c_meta_init = _sig("lnfp8_meta_init", [C.POINTER(CMeta), _P])
_c_update = _sig("amax_history_update", [C.POINTER(CMeta), C.POINTER(CRecipe), C.POINTER(C.c_int), _P, _P])
_c_update_many = _sig("amax_history_update_many", [C.POINTER(CMeta), C.c_int, C.POINTER(CRecipe), C.POINTER(C.c_int),
                                                   C.POINTER(_P), _P])
_c_quant = _sig("fp8_quantize", [_P, C.c_int, _I64, _I64, C.c_int, _P, _P, _P, _P, _P, _P])
_c_wquant = _sig("fp8_weight_quantize", [_P, _I64, _I64, C.POINTER(CMeta), C.POINTER(CRecipe), C.c_int, _P, _P])
_c_ln_fwd = _sig("ln_fwd_cast", [_P, _P, _P, C.c_float, _I64, _I64, C.c_int, _P, _P, _P, _P, _P, _P, _P])
_c_ln_bwd = _sig("ln_bwd", [_P, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P])
_c_gemm = _sig("fp8_gemm", [_P, C.c_int, C.c_int, _P, C.c_int, C.c_int, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I64,
                            _P])
_c_gemm_ws = _sig("lnfp8_gemm_workspace_size", [_I64, _I64, _I64], C.c_int64)
_c_lin_bwd_ws = _sig("lnfp8_ln_linear_bwd_workspace_size", [_I64, _I64, _I64], C.c_int64)
_c_mlp_bwd_ws = _sig("lnfp8_ln_mlp_bwd_workspace_size", [_I64, _I64, _I64], C.c_int64)
_c_mlp_fwd_ws = _sig("lnfp8_ln_mlp_fwd_workspace_size", [_I64, _I64, _I64], C.c_int64)
_c_ctx_bytes = _sig("lnfp8_ctx_bytes", [C.c_int, _I64, _I64, _I64], C.c_int64)
_c_ctx_offsets = _sig("lnfp8_ctx_offsets", [C.c_int, _I64, _I64, _I64, C.POINTER(_I64), C.c_int], C.c_int)
_c_lin_fwd = _sig("ln_linear_fwd", [C.POINTER(CLnLinearFwd), _P])
_c_lin_bwd = _sig("ln_linear_bwd", [C.POINTER(CLnLinearBwd), _P])
_c_lin_bwd_noalloc = _sig("ln_linear_bwd_noalloc", [C.POINTER(CLnLinearBwd), _P])
_c_mlp_fwd = _sig("ln_mlp_fwd", [C.POINTER(CLnMlpFwd), _P])
_c_mlp_bwd = _sig("ln_mlp_bwd", [C.POINTER(CLnMlpBwd), _P])


def _check(st: int) -> None:
    if st != OK:
        raise LnFp8Error(st, _lib.lnfp8_last_error().decode())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def version() -> int:
    return _c_version()


def last_error() -> str:
    return _lib.lnfp8_last_error().decode()


def lnfp8_selftest_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait diagnostic; the next sync_status() raises ERR_TIMEOUT."""
    _check(_c_selftest(int(limit_ns), _stream(stream)))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(_c_launch_count())


def profile_enable(on: bool = True) -> None:
    """Per-kernel CUDA-event timing on the launching stream (discards old records)."""
    _check(_c_prof_enable(int(on)))


def profile_sample() -> None:
    """After a replay of a graph captured with profiling on: add its kernel times to the totals."""
    _check(_c_prof_sample())


def profile_collect() -> dict:
    """{kernel kind: (total_ms, launches)} for everything recorded since profile_enable."""
    n = _c_prof_collect()
    out = {}
    for i in range(n):
        k, ms, cnt = C.c_char_p(), C.c_double(), C.c_longlong()
        _check(_c_prof_get(i, C.byref(k), C.byref(ms), C.byref(cnt)))
        out[k.value.decode()] = (ms.value, cnt.value)
    return out


def sync_status(stream=None) -> None:
    """Synchronise and raise if a bounded device wait has given up since the last check."""
    _check(_c_sync(_stream(stream)))


# ------------------------------------------------------------------ state
@dataclass
class Recipe:
    """DelayedScaling(fp8_format, amax_history_len, amax_compute_algo) of the TE tutorial."""
    fp8_format: str = "hybrid"
    amax_history_len: int = 16
    amax_compute_algo: str = "max"
    margin: int = 0

    def c(self) -> CRecipe:
        if self.amax_compute_algo != "max":
            raise ValueError("only amax_compute_algo='max' is supported")
        return CRecipe(_FORMATS[self.fp8_format], self.amax_history_len, 0, self.margin)

    @property
    def fwd_dtype(self) -> int:
        return E5M2 if self.fp8_format == "e5m2" else E4M3

    @property
    def bwd_dtype(self) -> int:
        return E4M3 if self.fp8_format == "e4m3" else E5M2


class ScalingMeta:
    """Device-resident delayed-scaling state of n FP8 tensors (one fp8_meta
    direction): scale [n], scale_inv [n], amax_history [L, n], amax_cur [n]."""

    def __init__(self, n: int, history_len: int, device="cuda", stream=None):
        self.n, self.history_len = n, history_len
        self.scale = torch.empty(n, dtype=torch.float32, device=device)
        self.scale_inv = torch.empty(n, dtype=torch.float32, device=device)
        self.amax_history = torch.empty(history_len, n, dtype=torch.float32, device=device)
        self.amax_cur = torch.empty(n, dtype=torch.float32, device=device)
        lnfp8_meta_init(self, stream)

    def c(self) -> CMeta:
        return CMeta(self.scale.data_ptr(), self.scale_inv.data_ptr(), self.amax_history.data_ptr(),
                     self.amax_cur.data_ptr(), self.n, self.history_len)

    def state_dict(self) -> dict:
        return {k: getattr(self, k).clone() for k in ("scale", "scale_inv", "amax_history", "amax_cur")}

    def load_state_dict(self, sd: dict) -> None:
        for k in ("scale", "scale_inv", "amax_history", "amax_cur"):
            getattr(self, k).copy_(sd[k])


def lnfp8_meta_init(meta: ScalingMeta, stream=None) -> None:
    cm = meta.c()
    _check(_c_meta_init(C.byref(cm), _stream(stream)))


def amax_history_update(meta: ScalingMeta, recipe: Recipe, dtypes, scale_inv_before=None, stream=None) -> None:
    arr = (C.c_int * meta.n)(*[int(d) for d in dtypes])
    cm, cr = meta.c(), recipe.c()
    _check(_c_update(C.byref(cm), C.byref(cr), arr, _ptr(scale_inv_before), _stream(stream)))


# ------------------------------------------------------------------ kernels

def amax_history_update_many(metas, recipe: Recipe, dtypes_per_meta, scale_inv_before=None, stream=None) -> None:
    """One launch of the state update for several ScalingMeta sets (e.g. all layers after a step)."""
    metas = list(metas)
    arr = (CMeta * len(metas))(*[m.c() for m in metas])
    flat = [int(d) for ds in dtypes_per_meta for d in ds]
    if len(flat) != sum(m.n for m in metas):
        raise ValueError("one dtype per slot of every meta")
    dts = (C.c_int * max(len(flat), 1))(*flat)
    sinv = None
    if scale_inv_before is not None:
        sinv = (_P * len(metas))(*[_ptr(t) for t in scale_inv_before])
    rc = recipe.c()
    _check(_c_update_many(arr, len(metas), C.byref(rc), dts, sinv, _stream(stream)))

def fp8_quantize(x, dtype, scale, amax_cur, *, out=None, out_t=None, colsum=None, stream=None):
    """codes = fp8(x * scale) with amax; x is a 2-D bf16 or fp32 CUDA tensor."""
    rows, cols = x.shape
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("fp8_quantize takes bf16 or fp32 input")
    _check(_c_quant(_ptr(x), int(x.dtype == torch.float32), rows, cols, dtype, _ptr(scale), _ptr(amax_cur),
                    _ptr(out), _ptr(out_t), _ptr(colsum), _stream(stream)))
    return out, out_t, colsum


@dataclass
class FP8Weight:
    """A weight kept as FP8 codes (fp8_model_init): codes [rows, cols] uint8 in the
    recipe's forward format, and the weight's own state (n = 1), whose scale_inv
    [1] is the codes' dequantisation factor."""
    codes: torch.Tensor
    meta: "ScalingMeta"
    dtype: int

    @property
    def scale_inv(self) -> torch.Tensor:
        return self.meta.scale_inv

    @property
    def shape(self):
        return self.codes.shape


def quantize_weight(w, recipe: Recipe, *, meta: ScalingMeta | None = None, codes=None, stream=None) -> FP8Weight:
    """Converts a bf16 weight [rows, cols] to FP8 storage once, on the device: its
    amax, the delayed-scaling state update of its own state, then the cast."""
    rows, cols = w.shape
    if w.dtype != torch.bfloat16:
        raise TypeError("quantize_weight takes a bf16 weight")
    meta = meta if meta is not None else ScalingMeta(1, 1, device=w.device, stream=stream)
    codes = codes if codes is not None else _e((rows, cols), torch.uint8, w.device)
    dt = recipe.fwd_dtype
    cm, cr = meta.c(), recipe.c()
    _check(_c_wquant(_ptr(w), rows, cols, C.byref(cm), C.byref(cr), dt, _ptr(codes), _stream(stream)))
    return FP8Weight(codes=codes, meta=meta, dtype=dt)


def ln_fwd_cast(x, gamma, beta, dtype, scale, amax_cur, *, eps=1e-5, out=None, mu=None, rsigma=None, y_debug=None,
                stream=None):
    M, D = x.shape
    dev = x.device
    out = out if out is not None else torch.empty(M, D, dtype=torch.uint8, device=dev)
    mu = mu if mu is not None else torch.empty(M, dtype=torch.float32, device=dev)
    rsigma = rsigma if rsigma is not None else torch.empty(M, dtype=torch.float32, device=dev)
    _check(_c_ln_fwd(_ptr(x), _ptr(gamma), _ptr(beta), eps, M, D, dtype, _ptr(scale), _ptr(amax_cur), _ptr(out),
                     _ptr(mu), _ptr(rsigma), _ptr(y_debug), _stream(stream)))
    return out, mu, rsigma


def ln_bwd(dy, x, gamma, mu, rsigma, *, dx=None, dgamma=None, dbeta=None, stream=None):
    M, D = x.shape
    dev = x.device
    dx = dx if dx is not None else torch.empty(M, D, dtype=torch.bfloat16, device=dev)
    dgamma = dgamma if dgamma is not None else torch.empty(D, dtype=torch.float32, device=dev)
    dbeta = dbeta if dbeta is not None else torch.empty(D, dtype=torch.float32, device=dev)
    _check(_c_ln_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mu), _ptr(rsigma), M, D, _ptr(dx), _ptr(dgamma),
                     _ptr(dbeta), _stream(stream)))
    return dx, dgamma, dbeta


def gemm_workspace_size(M, N, K) -> int:
    """Bytes of workspace with which fp8_gemm splits K for this shape (0: it would not)."""
    return int(_c_gemm_ws(M, N, K))


def ln_linear_bwd_workspace_size(M, K, N) -> int:
    return int(_c_lin_bwd_ws(M, K, N))


def ln_mlp_bwd_workspace_size(M, D, F) -> int:
    return int(_c_mlp_bwd_ws(M, D, F))


def ln_mlp_fwd_workspace_size(M, D, F) -> int:
    return int(_c_mlp_fwd_ws(M, D, F))


def _ws(nbytes, device):
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes > 0 else None


def fp8_gemm(a, a_layout, a_dtype, b, b_layout, b_dtype, M, N, K, sinv_a, sinv_b, *, bias=None, out=None,
             workspace=None, stream=None):
    """out[M, N] bf16 = (A . B^T) * sinv_a * sinv_b + bias; layouts as in the C ABI. With a
    uint8 workspace tensor of gemm_workspace_size(M, N, K) bytes the GEMM may split K."""
    out = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=b.device)
    _check(_c_gemm(_ptr(a), a_layout, a_dtype, _ptr(b), b_layout, b_dtype, M, N, K, _ptr(sinv_a), _ptr(sinv_b),
                   _ptr(bias), _ptr(out), _ptr(workspace), workspace.numel() if workspace is not None else 0,
                   _stream(stream)))
    return out


# ------------------------------------------------------------------ modules
@dataclass
class LinearCtx:
    xq: torch.Tensor
    wq: torch.Tensor
    mu: torch.Tensor | None
    rsigma: torch.Tensor | None
    sinv_saved: torch.Tensor
    ln_out_debug: torch.Tensor | None = None
    x_sum: torch.Tensor | None = None  # h = bf16(x + residual) of a forward with a residual (the backward's x)


def _e(shape, dtype, dev):
    return torch.empty(shape, dtype=dtype, device=dev)


def ctx_bytes(op: int, M: int, D: int, F: int) -> int:
    return int(_c_ctx_bytes(op, M, D, F))


def ctx_offsets(op: int, M: int, D: int, F: int) -> list:
    """Start of each saved-context buffer, then the total (the library's layout)."""
    off = (_I64 * 9)()
    n = int(_c_ctx_offsets(op, M, D, F, off, 9))
    if n < 0:
        raise LnFp8Error(ERR_INVALID_ARG, f"lnfp8_ctx_offsets({op}, {M}, {D}, {F})")
    return [int(off[i]) for i in range(n + 1)]


def _carve(op, M, D, F, shapes, device):
    """The saved context as views of one allocation laid out by lnfp8_ctx_offsets;
    shapes: (shape, dtype) per buffer in the library's order."""
    off = ctx_offsets(op, M, D, F)
    buf = torch.empty(off[-1], dtype=torch.uint8, device=device)
    views = []
    for (shape, dtype), start in zip(shapes, off):
        nbytes = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        views.append(buf[start:start + nbytes].view(dtype).view(shape))
    return buf, views


def linear_ctx(M, K, N, *, ln=True, device="cuda", debug=False, weight_codes=True) -> LinearCtx:
    """Saved tensors of one LayerNormLinear / Linear forward, views of one allocation in
    the library's saved-context layout (weight_codes=False leaves wq to an FP8Weight)."""
    u8, f32 = torch.uint8, torch.float32
    if ln:
        _, (xq, wq, mu, rs, sinv) = _carve(OP_LN_LINEAR, M, K, N, [((M, K), u8), ((N, K), u8), ((M,), f32),
                                                                   ((M,), f32), ((2,), f32)], device)
    else:
        _, (xq, wq, sinv) = _carve(OP_LINEAR, M, K, N, [((M, K), u8), ((N, K), u8), ((2,), f32)], device)
        mu = rs = None
    return LinearCtx(xq=xq, wq=wq if weight_codes else None, mu=mu, rsigma=rs, sinv_saved=sinv,
                     ln_out_debug=_e((M, K), torch.float32, device) if debug else None)


def ln_linear_fwd(x, gamma, beta, w, bias, meta: ScalingMeta, recipe: Recipe, *, eps=1e-5, y=None,
                  ctx: LinearCtx | None = None, defer_update=False, debug=False, residual=None, path=PATH_AUTO,
                  stream=None):
    """LayerNormLinear (gamma given) or Linear (gamma None) forward; returns (y, ctx).
    w is a bf16 weight (cast every call) or an FP8Weight (its codes are used as they are).
    residual: optional bf16 [M, K]; the input becomes h = bf16(x + residual), returned as
    ctx.x_sum (pass it as the backward's x). path: PATH_AUTO, PATH_FUSED (one launch for
    the LayerNorm, casts and GEMM; K <= 768) or PATH_SEPARATE."""
    M, K = x.shape
    N = w.shape[0]
    dev = x.device
    w8 = isinstance(w, FP8Weight)
    ctx = ctx if ctx is not None else linear_ctx(M, K, N, ln=gamma is not None, device=dev, debug=debug,
                                                 weight_codes=not w8)
    if w8:
        ctx.wq = w.codes
    if residual is not None and ctx.x_sum is None:
        ctx.x_sum = _e((M, K), torch.bfloat16, dev)
    y = y if y is not None else _e((M, N), torch.bfloat16, dev)
    a = CLnLinearFwd(M=M, K=K, N=N, x=_ptr(x), gamma=_ptr(gamma), beta=_ptr(beta), eps=eps,
                     w=None if w8 else _ptr(w), bias=_ptr(bias), y=_ptr(y), xq=_ptr(ctx.xq), wq=_ptr(ctx.wq),
                     mu=_ptr(ctx.mu), rsigma=_ptr(ctx.rsigma), sinv_saved=_ptr(ctx.sinv_saved), meta=meta.c(),
                     recipe=recipe.c(), defer_update=int(defer_update), ln_out_debug=_ptr(ctx.ln_out_debug),
                     w_scale_inv=_ptr(w.scale_inv) if w8 else None, residual=_ptr(residual),
                     x_sum=_ptr(ctx.x_sum) if residual is not None else None, path=int(path))
    _check(_c_lin_fwd(C.byref(a), _stream(stream)))
    return y, ctx


@dataclass
class LinearGrads:
    dx: torch.Tensor
    dw: torch.Tensor
    dbias: torch.Tensor | None
    dgamma: torch.Tensor | None
    dbeta: torch.Tensor | None
    dyq: torch.Tensor
    dln: torch.Tensor | None
    gemm_ws: torch.Tensor | None = None  # split-K workspace of the GEMMs (None: unsplit)


def linear_grads(M, K, N, *, ln=True, bias=True, split_k=True, device="cuda") -> LinearGrads:
    return LinearGrads(dx=_e((M, K), torch.bfloat16, device), dw=_e((N, K), torch.bfloat16, device),
                       dbias=_e((N,), torch.float32, device) if bias else None,
                       dgamma=_e((K,), torch.float32, device) if ln else None,
                       dbeta=_e((K,), torch.float32, device) if ln else None,
                       dyq=_e((M, N), torch.uint8, device), dln=_e((M, K), torch.bfloat16, device) if ln else None,
                       gemm_ws=_ws(ln_linear_bwd_workspace_size(M, K, N), device) if split_k else None)


def ln_linear_bwd(dy, x, gamma, ctx: LinearCtx, meta: ScalingMeta, recipe: Recipe, *, grads: LinearGrads | None = None,
                  bias=True, defer_update=False, stream=None) -> LinearGrads:
    M, N = dy.shape
    K = x.shape[1]
    g = grads if grads is not None else linear_grads(M, K, N, ln=gamma is not None, bias=bias, device=dy.device)
    a = CLnLinearBwd(M=M, K=K, N=N, dy=_ptr(dy), x=_ptr(x), gamma=_ptr(gamma), xq=_ptr(ctx.xq), wq=_ptr(ctx.wq),
                     mu=_ptr(ctx.mu), rsigma=_ptr(ctx.rsigma), sinv_saved=_ptr(ctx.sinv_saved), dx=_ptr(g.dx),
                     dw=_ptr(g.dw), dbias=_ptr(g.dbias), dgamma=_ptr(g.dgamma), dbeta=_ptr(g.dbeta),
                     dyq=_ptr(g.dyq), dln=_ptr(g.dln), meta=meta.c(), recipe=recipe.c(),
                     defer_update=int(defer_update), gemm_ws=_ptr(g.gemm_ws),
                     gemm_ws_bytes=g.gemm_ws.numel() if g.gemm_ws is not None else 0)
    _check(_c_lin_bwd(C.byref(a), _stream(stream)))
    return g


def ln_linear_bwd_noalloc(dy, x, gamma, ctx: LinearCtx, meta: ScalingMeta, recipe: Recipe, *, dx, dw, dbias=None,
                          dgamma=None, dbeta=None, defer_update=False, stream=None) -> None:
    """LayerNormLinear backward for callers that cannot allocate device memory:
    the caller passes inputs and outputs only; the library's built-in scratch
    array holds the dY codes and the LayerNorm-output gradient (see the C
    header for its size limit and sharing rules)."""
    M, N = dy.shape
    K = x.shape[1]
    a = CLnLinearBwd(M=M, K=K, N=N, dy=_ptr(dy), x=_ptr(x), gamma=_ptr(gamma), xq=_ptr(ctx.xq), wq=_ptr(ctx.wq),
                     mu=_ptr(ctx.mu), rsigma=_ptr(ctx.rsigma), sinv_saved=_ptr(ctx.sinv_saved), dx=_ptr(dx),
                     dw=_ptr(dw), dbias=_ptr(dbias), dgamma=_ptr(dgamma), dbeta=_ptr(dbeta), dyq=None, dln=None,
                     meta=meta.c(), recipe=recipe.c(), defer_update=int(defer_update))
    _check(_c_lin_bwd_noalloc(C.byref(a), _stream(stream)))


@dataclass
class MlpCtx:
    lnq: torch.Tensor
    mu: torch.Tensor
    rsigma: torch.Tensor
    w1q: torch.Tensor
    w2q: torch.Tensor
    h: torch.Tensor
    aq: torch.Tensor
    sinv_saved: torch.Tensor
    ln_out_debug: torch.Tensor | None = None
    act_debug: torch.Tensor | None = None
    gemm_ws: torch.Tensor | None = None  # FC1 tiles' readiness counters (FC1 and FC2 in one launch)
    x_sum: torch.Tensor | None = None  # h = bf16(x + residual) of a forward with a residual (the backward's x)


def mlp_ctx(M, D, F, *, device="cuda", debug=False, fused=False, weight_codes=True) -> MlpCtx:
    """Saved tensors of one LayerNormMLP forward. fused=True also allocates the row-block
    readiness counters with which the forward runs FC1 and FC2 as one launch (same
    results; the two launches measured faster at 8192 x 768 -> 3072 -> 768 and at
    d 2048 from 8192 to 65536 tokens, equal at 2048).
    weight_codes=False leaves w1q/w2q to FP8-stored weights."""
    u8, f32 = torch.uint8, torch.float32
    _, (lnq, w1q, w2q, h, aq, mu, rs, sinv) = _carve(
        OP_LN_MLP, M, D, F, [((M, D), u8), ((F, D), u8), ((D, F), u8), ((M, F), torch.bfloat16), ((M, F), u8),
                             ((M,), f32), ((M,), f32), ((4,), f32)], device)
    return MlpCtx(lnq=lnq, mu=mu, rsigma=rs, w1q=w1q if weight_codes else None, w2q=w2q if weight_codes else None,
                  h=h, aq=aq, sinv_saved=sinv,
                  ln_out_debug=_e((M, D), torch.float32, device) if debug else None,
                  act_debug=_e((M, F), torch.float32, device) if debug else None,
                  gemm_ws=_ws(ln_mlp_fwd_workspace_size(M, D, F), device) if fused else None)


def ln_mlp_fwd(x, gamma, beta, w1, b1, w2, b2, meta: ScalingMeta, recipe: Recipe, *, eps=1e-5, y=None,
               ctx: MlpCtx | None = None, defer_update=False, debug=False, residual=None, stream=None):
    """LayerNormMLP forward; returns (y, ctx). w1 and w2 are both bf16 weights (cast
    every call) or both FP8Weight (their codes are used as they are). residual: optional
    bf16 [M, D]; the input becomes h = bf16(x + residual), returned as ctx.x_sum."""
    M, D = x.shape
    F = w1.shape[0]
    dev = x.device
    w8 = isinstance(w1, FP8Weight)
    if w8 != isinstance(w2, FP8Weight):
        raise TypeError("w1 and w2 must both be FP8Weight or both bf16")
    ctx = ctx if ctx is not None else mlp_ctx(M, D, F, device=dev, debug=debug, weight_codes=not w8)
    if w8:
        ctx.w1q, ctx.w2q = w1.codes, w2.codes
    if residual is not None and ctx.x_sum is None:
        ctx.x_sum = _e((M, D), torch.bfloat16, dev)
    y = y if y is not None else _e((M, D), torch.bfloat16, dev)
    a = CLnMlpFwd(M=M, D=D, F=F, x=_ptr(x), gamma=_ptr(gamma), beta=_ptr(beta), eps=eps,
                  w1=None if w8 else _ptr(w1), b1=_ptr(b1), w2=None if w8 else _ptr(w2), b2=_ptr(b2), y=_ptr(y),
                  lnq=_ptr(ctx.lnq), mu=_ptr(ctx.mu), rsigma=_ptr(ctx.rsigma),
                  w1q=_ptr(ctx.w1q), w2q=_ptr(ctx.w2q), h=_ptr(ctx.h), aq=_ptr(ctx.aq),
                  sinv_saved=_ptr(ctx.sinv_saved), meta=meta.c(), recipe=recipe.c(), defer_update=int(defer_update),
                  ln_out_debug=_ptr(ctx.ln_out_debug), act_debug=_ptr(ctx.act_debug), gemm_ws=_ptr(ctx.gemm_ws),
                  gemm_ws_bytes=ctx.gemm_ws.numel() if ctx.gemm_ws is not None else 0,
                  w1_scale_inv=_ptr(w1.scale_inv) if w8 else None, w2_scale_inv=_ptr(w2.scale_inv) if w8 else None,
                  residual=_ptr(residual), x_sum=_ptr(ctx.x_sum) if residual is not None else None)
    _check(_c_mlp_fwd(C.byref(a), _stream(stream)))
    return y, ctx


@dataclass
class MlpGrads:
    dx: torch.Tensor
    dgamma: torch.Tensor
    dbeta: torch.Tensor
    dw1: torch.Tensor
    db1: torch.Tensor | None
    dw2: torch.Tensor
    db2: torch.Tensor | None
    dyq: torch.Tensor
    dhq: torch.Tensor
    dln: torch.Tensor
    dh_debug: torch.Tensor | None = None
    gemm_ws: torch.Tensor | None = None  # split-K workspace of the GEMMs (None: unsplit)


def mlp_grads(M, D, F, *, bias=True, split_k=True, device="cuda", debug=False) -> MlpGrads:
    return MlpGrads(dx=_e((M, D), torch.bfloat16, device), dgamma=_e((D,), torch.float32, device),
                    dbeta=_e((D,), torch.float32, device), dw1=_e((F, D), torch.bfloat16, device),
                    db1=_e((F,), torch.float32, device) if bias else None, dw2=_e((D, F), torch.bfloat16, device),
                    db2=_e((D,), torch.float32, device) if bias else None, dyq=_e((M, D), torch.uint8, device),
                    dhq=_e((M, F), torch.uint8, device), dln=_e((M, D), torch.bfloat16, device),
                    dh_debug=_e((M, F), torch.float32, device) if debug else None,
                    gemm_ws=_ws(ln_mlp_bwd_workspace_size(M, D, F), device) if split_k else None)


def ln_mlp_bwd(dy, x, gamma, ctx: MlpCtx, meta: ScalingMeta, recipe: Recipe, *, grads: MlpGrads | None = None,
               bias=True, defer_update=False, debug=False, stream=None) -> MlpGrads:
    M, D = dy.shape
    F = ctx.h.shape[1]
    g = grads if grads is not None else mlp_grads(M, D, F, bias=bias, device=dy.device, debug=debug)
    a = CLnMlpBwd(M=M, D=D, F=F, dy=_ptr(dy), x=_ptr(x), gamma=_ptr(gamma), lnq=_ptr(ctx.lnq), mu=_ptr(ctx.mu),
                  rsigma=_ptr(ctx.rsigma), w1q=_ptr(ctx.w1q), w2q=_ptr(ctx.w2q), h=_ptr(ctx.h), aq=_ptr(ctx.aq),
                  sinv_saved=_ptr(ctx.sinv_saved), dx=_ptr(g.dx), dgamma=_ptr(g.dgamma), dbeta=_ptr(g.dbeta),
                  dw1=_ptr(g.dw1), db1=_ptr(g.db1), dw2=_ptr(g.dw2), db2=_ptr(g.db2), dyq=_ptr(g.dyq),
                  dhq=_ptr(g.dhq), dln=_ptr(g.dln), meta=meta.c(), recipe=recipe.c(),
                  defer_update=int(defer_update), dh_debug=_ptr(g.dh_debug), gemm_ws=_ptr(g.gemm_ws),
                  gemm_ws_bytes=g.gemm_ws.numel() if g.gemm_ws is not None else 0)
    _check(_c_mlp_bwd(C.byref(a), _stream(stream)))
    return g
