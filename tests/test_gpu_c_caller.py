"""A plain C program drives one LayerNormMLP step through the C ABI (GPU).

The program is C11 built on include/lnfp8.h and linked to liblnfp8.so and the
CUDA runtime; no Python or PyTorch is involved on its side. It allocates device
memory with cudaMalloc, carves the saved context out of one allocation at the
offsets lnfp8_ctx_offsets gives, initialises both states, runs ln_mlp_fwd and
ln_mlp_bwd on the default stream, checks lnfp8_sync_status, and writes the
outputs and the states to files. The test compares them with the oracle step
from the same inputs: bf16 outputs and gradients within 1e-2 relative
Frobenius error, the weight amaxes bit for bit.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from fp8_delayed_scaling_row_gb300 import synth
from oracle import fp8 as ofp8
from oracle import modules as omod
from oracle.delayed_scaling import Recipe, ScalingState
from oracle.gemm import bf16_to_f32
from helpers import rel_fro

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "lnfp8.h"

#define NM 300 /* tokens */
#define ND 256 /* hidden */
#define NF 512 /* FFN width */
#define NL 16  /* history length */

static void* dmalloc(size_t n) {
  void* p = NULL;
  if (cudaMalloc(&p, n ? n : 16) != cudaSuccess) { fprintf(stderr, "cudaMalloc failed\n"); exit(2); }
  return p;
}
static void load(const char* dir, const char* name, void* dev, size_t n) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s.bin", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "missing %s\n", path); exit(2); }
  void* h = malloc(n);
  if (fread(h, 1, n, f) != n) { fprintf(stderr, "short %s\n", path); exit(2); }
  fclose(f);
  cudaMemcpy(dev, h, n, cudaMemcpyHostToDevice);
  free(h);
}
static void save(const char* dir, const char* name, const void* dev, size_t n) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s.out", dir, name);
  void* h = malloc(n);
  cudaMemcpy(h, dev, n, cudaMemcpyDeviceToHost);
  FILE* f = fopen(path, "wb");
  fwrite(h, 1, n, f);
  fclose(f);
  free(h);
}
static lnfp8_meta meta(int n) {
  lnfp8_meta m;
  m.scale = (float*)dmalloc(4 * n);
  m.scale_inv = (float*)dmalloc(4 * n);
  m.amax_history = (float*)dmalloc(4 * n * NL);
  m.amax_cur = (float*)dmalloc(4 * n);
  m.n = n;
  m.history_len = NL;
  return m;
}
#define TRY(x) do { lnfp8_status s_ = (x); if (s_ != LNFP8_OK) { fprintf(stderr, "%s -> %d: %s\n", #x, (int)s_, lnfp8_last_error()); return 1; } } while (0)

int main(int argc, char** argv) {
  const char* dir = argv[1];
  uint16_t *x = dmalloc(2 * NM * ND), *dy = dmalloc(2 * NM * ND), *gamma = dmalloc(2 * ND), *beta = dmalloc(2 * ND);
  uint16_t *w1 = dmalloc(2 * NF * ND), *b1 = dmalloc(2 * NF), *w2 = dmalloc(2 * ND * NF), *b2 = dmalloc(2 * ND);
  load(dir, "x", x, 2 * NM * ND); load(dir, "dy", dy, 2 * NM * ND); load(dir, "gamma", gamma, 2 * ND);
  load(dir, "beta", beta, 2 * ND); load(dir, "w1", w1, 2 * NF * ND); load(dir, "b1", b1, 2 * NF);
  load(dir, "w2", w2, 2 * ND * NF); load(dir, "b2", b2, 2 * ND);
  /* the saved context: one allocation, the library's layout */
  int64_t off[9];
  if (lnfp8_ctx_offsets(LNFP8_OP_LN_MLP, NM, ND, NF, off, 9) != 8) return 1;
  unsigned char* ctx = dmalloc((size_t)off[8]);
  lnfp8_meta fm = meta(4), bm = meta(2);
  lnfp8_recipe rec = {LNFP8_FORMAT_HYBRID, NL, 0, 0};
  TRY(lnfp8_meta_init(&fm, NULL));
  TRY(lnfp8_meta_init(&bm, NULL));
  lnfp8_ln_mlp_fwd_args a;
  memset(&a, 0, sizeof a);
  a.M = NM; a.D = ND; a.F = NF; a.x = x; a.gamma = gamma; a.beta = beta; a.eps = 1e-5f;
  a.w1 = w1; a.b1 = b1; a.w2 = w2; a.b2 = b2;
  a.y = dmalloc(2 * NM * ND);
  a.lnq = ctx + off[0]; a.w1q = ctx + off[1]; a.w2q = ctx + off[2]; a.h = (uint16_t*)(ctx + off[3]);
  a.aq = ctx + off[4]; a.mu = (float*)(ctx + off[5]); a.rsigma = (float*)(ctx + off[6]);
  a.sinv_saved = (float*)(ctx + off[7]);
  a.meta = fm; a.recipe = rec;
  TRY(ln_mlp_fwd(&a, NULL));
  lnfp8_ln_mlp_bwd_args g;
  memset(&g, 0, sizeof g);
  g.M = NM; g.D = ND; g.F = NF; g.dy = dy; g.x = x; g.gamma = gamma;
  g.lnq = a.lnq; g.mu = a.mu; g.rsigma = a.rsigma; g.w1q = a.w1q; g.w2q = a.w2q; g.h = a.h; g.aq = a.aq;
  g.sinv_saved = a.sinv_saved;
  g.dx = dmalloc(2 * NM * ND); g.dgamma = dmalloc(4 * ND); g.dbeta = dmalloc(4 * ND);
  g.dw1 = dmalloc(2 * NF * ND); g.db1 = dmalloc(4 * NF); g.dw2 = dmalloc(2 * ND * NF); g.db2 = dmalloc(4 * ND);
  g.dyq = dmalloc(NM * ND); g.dhq = dmalloc(NM * NF); g.dln = dmalloc(2 * NM * ND);
  g.meta = bm; g.recipe = rec;
  TRY(ln_mlp_bwd(&g, NULL));
  TRY(lnfp8_sync_status(NULL));
  save(dir, "y", a.y, 2 * NM * ND); save(dir, "dx", g.dx, 2 * NM * ND); save(dir, "dw1", g.dw1, 2 * NF * ND);
  save(dir, "dw2", g.dw2, 2 * ND * NF); save(dir, "db1", g.db1, 4 * NF); save(dir, "db2", g.db2, 4 * ND);
  save(dir, "dgamma", g.dgamma, 4 * ND); save(dir, "dbeta", g.dbeta, 4 * ND);
  save(dir, "fwd_history", fm.amax_history, 4 * 4 * NL); save(dir, "bwd_history", bm.amax_history, 4 * 2 * NL);
  printf("ok\n");
  return 0;
}
"""

M, D, F, HIST = 300, 256, 512, 16


def test_c_program_runs_a_layernorm_mlp_step(tmp_path):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    from fp8_delayed_scaling_row_gb300.build import LIB, build_library
    if not os.path.exists(LIB):
        build_library()
    libdir = os.path.dirname(LIB)
    p = synth.mlp_params(D, F, seed=31, bias_std=0.02)
    x = synth.activations(M, D, dist="outliers", seed=31)
    dy = synth.grad(M, D, seed=31)
    for name, bits in dict(p, x=x, dy=dy).items():
        np.ascontiguousarray(bits, dtype=np.uint16).tofile(tmp_path / f"{name}.bin")
    src, exe = tmp_path / "mlp_step.c", tmp_path / "mlp_step"
    src.write_text(PROGRAM)
    cudalib = os.path.join(CUDA, "lib64")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wno-pointer-sign", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(CUDA, "include"), str(src), "-o", str(exe), "-L", libdir, "-l:liblnfp8.so",
                    "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"], check=True)
    out = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr

    def rd(name, dtype, shape):
        a = np.fromfile(tmp_path / f"{name}.out", dtype=dtype).reshape(shape)
        return bf16_to_f32(a).astype(np.float64) if dtype == np.uint16 else a.astype(np.float64)

    rec = Recipe("hybrid", HIST)
    fs, bs = ScalingState(4, HIST), ScalingState(2, HIST)
    Y, ctx, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs, rec)
    og = omod.ln_mlp_bwd(dy, ctx, bs, rec)
    assert rel_fro(rd("y", np.uint16, (M, D)), Y) < 1e-2
    for k, dt, shape in [("dx", np.uint16, (M, D)), ("dw1", np.uint16, (F, D)), ("dw2", np.uint16, (D, F)),
                         ("db1", np.float32, (F,)), ("db2", np.float32, (D,)), ("dgamma", np.float32, (D,)),
                         ("dbeta", np.float32, (D,))]:
        assert rel_fro(rd(k, dt, shape), og[k]) < 1e-2, k
    fh = np.fromfile(tmp_path / "fwd_history.out", dtype=np.float32).reshape(HIST, 4)
    bh = np.fromfile(tmp_path / "bwd_history.out", dtype=np.float32).reshape(HIST, 2)
    assert fh[0, 1] == ofp8.amax(bf16_to_f32(p["w1"])) and fh[0, 3] == ofp8.amax(bf16_to_f32(p["w2"]))
    assert bh[0, 0] == ofp8.amax(bf16_to_f32(dy))
    # amaxes of computed tensors: LN output within 2e-3, GELU output and dH within 1e-2 of the oracle's
    assert abs(float(fh[0, 0]) - float(fs.amax_history[0, 0])) <= 2e-3 * float(fs.amax_history[0, 0])
    assert abs(float(fh[0, 2]) - float(fs.amax_history[0, 2])) <= 1e-2 * float(fs.amax_history[0, 2])
    assert abs(float(bh[0, 1]) - float(bs.amax_history[0, 1])) <= 1e-2 * float(bs.amax_history[0, 1])
