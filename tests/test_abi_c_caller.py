"""The C ABI used from plain C (CPU): a C11 program built against
include/lnfp8.h and linked to liblnfp8.so calls the size queries and the
argument checks that answer before anything reaches the GPU, and reads the
error message of the last failing call."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lnfp8.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main(void) {
  CHECK(lnfp8_version() == 400);
  /* the saved-context layout: buffers at multiples of 256 bytes, then the total */
  int64_t off[9];
  CHECK(lnfp8_ctx_offsets(LNFP8_OP_LN_MLP, 300, 64, 128, off, 9) == 8);
  CHECK(off[0] == 0 && off[1] == 19200 && off[2] == 19200 + 8192 && off[8] == lnfp8_ctx_bytes(LNFP8_OP_LN_MLP, 300, 64, 128));
  CHECK(lnfp8_ctx_offsets(LNFP8_OP_LN_MLP, 300, 64, 128, off, 8) == -1);
  CHECK(lnfp8_ctx_bytes(7, 1, 16, 16) == -1 && lnfp8_ctx_bytes(LNFP8_OP_LINEAR, -1, 16, 16) == -1);
  /* size queries: pure host arithmetic */
  CHECK(lnfp8_ln_mlp_fwd_workspace_size(8192, 768, 3072) == 256);
  CHECK(lnfp8_ln_mlp_fwd_workspace_size(0, 768, 3072) == 0);
  CHECK(lnfp8_ln_mlp_fwd_workspace_size(-1, 768, 3072) == -1);
  CHECK(lnfp8_gemm_workspace_size(-1, 16, 16) == -1);
  CHECK(lnfp8_ln_mlp_bwd_workspace_size(8192, 768, 3072) >= 0);
  /* argument errors come back synchronously, with a message */
  float* fake = (float*)(size_t)0x10000;
  CHECK(fp8_quantize(fake, 0, 10, 24, LNFP8_E4M3, fake, fake, NULL, NULL, NULL, NULL) == LNFP8_ERR_UNSUPPORTED_SHAPE);
  CHECK(strstr(lnfp8_last_error(), "fp8_quantize") != NULL);
  CHECK(fp8_quantize(fake, 0, 10, 32, 7, fake, fake, NULL, NULL, NULL, NULL) == LNFP8_ERR_INVALID_ARG);
  lnfp8_ln_mlp_fwd_args a;
  memset(&a, 0, sizeof a);
  a.M = 64; a.D = 256; a.F = 512;
  CHECK(ln_mlp_fwd(&a, NULL) == LNFP8_ERR_INVALID_ARG); /* no state */
  CHECK(ln_mlp_fwd(NULL, NULL) == LNFP8_ERR_INVALID_ARG);
  lnfp8_meta m = {fake, fake, fake, fake, 2, 16};
  lnfp8_meta twice[2] = {m, m};
  lnfp8_recipe r = {LNFP8_FORMAT_HYBRID, 16, 0, 0};
  int dts[4] = {LNFP8_E4M3, LNFP8_E4M3, LNFP8_E4M3, LNFP8_E4M3};
  CHECK(amax_history_update_many(twice, 2, &r, dts, NULL, NULL) == LNFP8_ERR_INVALID_ARG);
  CHECK(amax_history_update_many(twice, 0, &r, dts, NULL, NULL) == LNFP8_OK); /* nothing to do */
  printf("ok\n");
  return 0;
}
"""


def test_c_program_calls_the_library():
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from fp8_delayed_scaling_row_gb300.build import LIB, build_library
    if not os.path.exists(LIB):
        build_library()
    libdir = os.path.dirname(LIB)
    d = os.path.join(ROOT, "tests", "__pycache__")
    os.makedirs(d, exist_ok=True)
    src, exe = os.path.join(d, "c_caller.c"), os.path.join(d, "c_caller")
    with open(src, "w") as f:
        f.write(PROGRAM)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-I", os.path.join(ROOT, "include"), src, "-o", exe, "-L", libdir,
                    "-l:liblnfp8.so", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr
