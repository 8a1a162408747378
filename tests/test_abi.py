"""The C ABI: the library loads and exports every entry point the header
declares, and argument errors come back synchronously, before anything is
enqueued (CPU only: no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lnfp8.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_delayed_scaling_row_gb300.build import LIB, build_library
    if not os.path.exists(LIB):
        build_library()
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:long\s+long|[a-z_0-9]+)\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("ln_linear_fwd", "ln_linear_bwd", "ln_mlp_fwd", "ln_mlp_bwd", "fp8_quantize", "amax_history_update"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    assert sorted(lib.EXPORTED) == declared_functions()


def test_version(lib):
    assert lib.version() == 400


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _meta(n, L):
    return lib_mod().CMeta(FAKE, FAKE, FAKE, FAKE, n, L)


def lib_mod():
    from fp8_delayed_scaling_row_gb300 import lnfp8
    return lnfp8


def _mlp_args(lnfp8, **kw):
    a = lnfp8.CLnMlpFwd(M=64, D=256, F=512, x=FAKE, gamma=FAKE, beta=FAKE, eps=1e-5, w1=FAKE, b1=None, w2=FAKE,
                        b2=None, y=FAKE, lnq=FAKE, mu=FAKE, rsigma=FAKE, w1q=FAKE, w2q=FAKE, h=FAKE, aq=FAKE,
                        sinv_saved=FAKE, meta=_meta(4, 16), recipe=lnfp8.CRecipe(1, 16, 0, 0), defer_update=0)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status,needle", [
    ("D", 100, 2, "multiple of 16"),
    ("F", 0, 2, "multiple of 16"),
    ("M", -1, 1, "M = -1"),
    ("D", 16384, 2, "D > 8192"),
    ("gamma", None, 1, "gamma is NULL"),
    ("w1", FAKE + 8, 1, "not 16-byte aligned"),
])
def test_mlp_fwd_rejects_bad_arguments(lib, field, value, status, needle):
    a = _mlp_args(lib, **{field: value})
    st = lib._c_mlp_fwd(ctypes.byref(a), None)
    assert st == status
    assert needle in lib.last_error()


def test_mlp_fwd_rejects_bad_meta_and_recipe(lib):
    a = _mlp_args(lib, meta=_meta(3, 16))
    assert lib._c_mlp_fwd(ctypes.byref(a), None) == 1 and "meta.n" in lib.last_error()
    a = _mlp_args(lib, recipe=lib.CRecipe(1, 8, 0, 0))
    assert lib._c_mlp_fwd(ctypes.byref(a), None) == 1 and "history_len" in lib.last_error()
    a = _mlp_args(lib, recipe=lib.CRecipe(1, 16, 1, 0))
    assert lib._c_mlp_fwd(ctypes.byref(a), None) == 5
    a = _mlp_args(lib, recipe=lib.CRecipe(7, 16, 0, 0))
    assert lib._c_mlp_fwd(ctypes.byref(a), None) == 1


def test_quantize_and_gemm_reject_bad_shapes(lib):
    assert lib._c_quant(FAKE, 0, 10, 24, 0, FAKE, FAKE, FAKE, None, None, None) == 2
    assert lib._c_quant(FAKE, 0, 10, 32, 3, FAKE, FAKE, FAKE, None, None, None) == 1
    assert lib._c_quant(FAKE, 0, 10, 32, 0, None, FAKE, FAKE, None, None, None) == 1
    # A stored [K, M] needs M % 16 == 0
    assert lib._c_gemm(FAKE, 1, 0, FAKE, 0, 0, 100, 32, 32, FAKE, FAKE, None, FAKE, None, 0, None) == 2
    assert lib._c_gemm(FAKE, 0, 0, FAKE, 2, 0, 100, 32, 32, FAKE, FAKE, None, FAKE, None, 0, None) == 1
    assert lib._c_gemm(FAKE, 0, 0, FAKE, 0, 0, 100, 32, 0, FAKE, FAKE, None, FAKE, None, 0, None) == 2
    # a misaligned workspace and a negative workspace size are rejected before anything runs
    assert lib._c_gemm(FAKE, 0, 0, FAKE, 0, 0, 100, 32, 32, FAKE, FAKE, None, FAKE, FAKE + 4, 1 << 20, None) == 1
    assert lib._c_gemm(FAKE, 0, 0, FAKE, 0, 0, 100, 32, 32, FAKE, FAKE, None, FAKE, FAKE, -1, None) == 1


def test_workspace_size_queries(lib):
    """The size queries need no GPU; negative sizes give -1 and an empty problem needs none."""
    assert lib.gemm_workspace_size(-1, 32, 32) == -1
    assert lib.ln_linear_bwd_workspace_size(16, -1, 32) == -1
    assert lib.ln_mlp_bwd_workspace_size(16, 32, -5) == -1
    assert lib.gemm_workspace_size(0, 0, 0) == 0
    for f in (lib.gemm_workspace_size, lib.ln_linear_bwd_workspace_size, lib.ln_mlp_bwd_workspace_size):
        n = f(8192, 768, 3072)
        assert n >= 0 and n % 256 == 0


def test_state_update_rejects_bad_arguments(lib):
    m = _meta(2, 16)
    dts = (ctypes.c_int * 2)(0, 1)
    assert lib._c_update(ctypes.byref(m), ctypes.byref(lib.CRecipe(1, 4, 0, 0)), dts, None, None) == 1
    assert lib._c_update(ctypes.byref(m), ctypes.byref(lib.CRecipe(1, 16, 0, 0)), None, None, None) == 1
    bad = (ctypes.c_int * 2)(0, 5)
    assert lib._c_update(ctypes.byref(m), ctypes.byref(lib.CRecipe(1, 16, 0, 0)), bad, None, None) == 1
    m0 = _meta(0, 16)
    assert lib._c_meta_init(ctypes.byref(m0), None) == 1
    assert lib._c_selftest(10, None) == 1


def test_update_many_and_new_entry_points_reject_bad_arguments(lib):
    rec = lib.CRecipe(1, 16, 0, 0)
    a, b = lib.CMeta(FAKE, FAKE, FAKE, FAKE, 2, 16), lib.CMeta(FAKE + 256, FAKE + 256, FAKE + 256, FAKE + 256, 2, 16)
    dts = (ctypes.c_int * 6)(0, 0, 0, 0, 0, 0)
    # the same set twice would have two CTAs update one slot
    arr = (lib.CMeta * 3)(a, b, a)
    assert lib._c_update_many(arr, 3, ctypes.byref(rec), dts, None, None) == 1 and "share state" in lib.last_error()
    # overlapping amax_cur ranges
    c = lib.CMeta(FAKE + 512, FAKE + 512, FAKE + 512, FAKE + 4, 2, 16)
    arr = (lib.CMeta * 2)(a, c)
    assert lib._c_update_many(arr, 2, ctypes.byref(rec), dts, None, None) == 1
    assert lib._c_update_many(arr, 129, ctypes.byref(rec), dts, None, None) == 1
    assert lib._c_update_many(arr, -1, ctypes.byref(rec), dts, None, None) == 1
    bad = (ctypes.c_int * 4)(0, 7, 0, 0)  # not an FP8 dtype
    arr = (lib.CMeta * 2)(a, b)
    assert lib._c_update_many(arr, 2, ctypes.byref(rec), bad, None, None) == 1
    # the weight conversion takes a one-slot state
    assert lib._c_wquant(FAKE, 64, 32, ctypes.byref(a), ctypes.byref(rec), 0, FAKE, None) == 1
    # a residual needs the LayerNorm it precedes
    la = lib.CLnLinearFwd(M=64, K=256, N=512, x=FAKE, gamma=None, beta=None, eps=1e-5, w=FAKE, bias=None, y=FAKE,
                          xq=FAKE, wq=FAKE, mu=None, rsigma=None, sinv_saved=FAKE, meta=lib.CMeta(FAKE, FAKE, FAKE, FAKE, 2, 16),
                          recipe=rec, defer_update=0, residual=FAKE, x_sum=FAKE)
    assert lib._c_lin_fwd(ctypes.byref(la), None) == 1 and "residual" in lib.last_error()
    # FP8 weights of an MLP come in pairs
    m = _mlp_args(lib, w1_scale_inv=FAKE)
    assert lib._c_mlp_fwd(ctypes.byref(m), None) == 1 and "together" in lib.last_error()


def test_saved_context_layout_by_hand(lib):
    # LayerNormMLP, M = 300 tokens, D = 64, F = 128: lnq 19200 B, w1q 8192, w2q 8192, h 76800, aq 38400,
    # mu 1200, rsigma 1200, sinv 16; each starts at a multiple of 256
    off = lib.ctx_offsets(lib.OP_LN_MLP, 300, 64, 128)
    sizes = [19200, 8192, 8192, 76800, 38400, 1200, 1200, 16]
    want, o = [], 0
    for n in sizes:
        want.append(o)
        o += (n + 255) // 256 * 256
    assert off == want + [o] and lib.ctx_bytes(lib.OP_LN_MLP, 300, 64, 128) == o == 153600
    # LayerNormLinear 768 -> 2304 over 256 tokens: xq, wq, mu, rsigma, sinv
    assert lib.ctx_offsets(lib.OP_LN_LINEAR, 256, 768, 2304) == [0, 196608, 196608 + 1769472, 196608 + 1769472 + 1024,
                                                               196608 + 1769472 + 2048, 196608 + 1769472 + 2304]
    assert lib.ctx_offsets(lib.OP_LINEAR, 0, 16, 32) == [0, 0, 512, 768]
    assert lib.ctx_bytes(5, 1, 16, 16) == -1 and lib.ctx_bytes(lib.OP_LN_MLP, 1, -16, 16) == -1
    with pytest.raises(lib.LnFp8Error):
        lib.ctx_offsets(9, 1, 16, 16)
