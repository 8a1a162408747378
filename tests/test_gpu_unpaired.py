"""The backward without the paired launches (GPU).

With LNFP8_NO_PAIR set (read once per process) each backward GEMM runs as its
own launch: the FC2 data gradient in gemm_kernel with its own dGELU epilogue,
the weight gradients as separate GEMMs. A child process runs one LayerNormMLP
backward that way; its dH codes and backward amaxes must equal the paired
launch's bit for bit (the same accumulators through the same dGELU arithmetic),
and the other outputs must agree up to fp32 summation order.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
from fp8_delayed_scaling_row_gb300 import lnfp8 as L, synth
from helpers import bf16_dev
M, D, F = int(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5])
p = {k: bf16_dev(v) for k, v in synth.mlp_params(D, F, seed=29, bias_std=0.02).items()}
x = bf16_dev(synth.activations(M, D, dist="outliers", seed=29, step=0))
dy = bf16_dev(synth.grad(M, D, seed=29, step=0))
rec = L.Recipe("hybrid", 4)
fm, bm = L.ScalingMeta(4, 4), L.ScalingMeta(2, 4)
ctx = L.mlp_ctx(M, D, F)
L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fm, rec, ctx=ctx)
g = L.ln_mlp_bwd(dy, x, p["gamma"], ctx, bm, rec)
L.sync_status()
out = {k: getattr(g, k).float().cpu().numpy() for k in ("dx", "dw1", "dw2", "db1", "db2", "dgamma", "dbeta", "dln")}
out["dhq"] = g.dhq.cpu().numpy()
out["bwd_hist"] = bm.amax_history.cpu().numpy()
np.savez(sys.argv[2], **out)
"""


@pytest.mark.parametrize("M,D,F", [(1000, 256, 1024), (8192, 768, 3072)])
def test_unpaired_backward_equals_the_paired_launches(tmp_path, M, D, F):
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    res = {}
    for tag, env in (("paired", {}), ("unpaired", {"LNFP8_NO_PAIR": "1"})):
        e = dict(os.environ, **env)
        e.pop("LNFP8_NO_PAIR", None) if not env else None
        out = tmp_path / f"{tag}.npz"
        r = subprocess.run([sys.executable, str(script), ROOT, str(out), str(M), str(D), str(F)], env=e,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout + r.stderr
        res[tag] = np.load(out)
    a, b = res["paired"], res["unpaired"]
    assert np.array_equal(a["dhq"], b["dhq"])
    assert np.array_equal(a["bwd_hist"].view(np.uint32), b["bwd_hist"].view(np.uint32))
    for k in ("dx", "dw1", "dw2", "db1", "db2", "dgamma", "dbeta", "dln"):
        x, y = a[k].astype(np.float64), b[k].astype(np.float64)
        assert np.linalg.norm(x - y) <= 1e-4 * np.linalg.norm(y), k
