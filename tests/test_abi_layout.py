"""The ctypes mirrors of the C-ABI structs have the header's layout: a small C
program built against include/lnfp8.h prints each struct's size and each
field's offset, and the Python binding's Structure classes must agree field by
field (names in header order, offsets, sizes)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lnfp8.h")

STRUCTS = {
    "lnfp8_recipe": "CRecipe",
    "lnfp8_meta": "CMeta",
    "lnfp8_ln_linear_fwd_args": "CLnLinearFwd",
    "lnfp8_ln_linear_bwd_args": "CLnLinearBwd",
    "lnfp8_ln_mlp_fwd_args": "CLnMlpFwd",
    "lnfp8_ln_mlp_bwd_args": "CLnMlpBwd",
}


def _header_fields():
    """Field names of each typedef'd struct, in declaration order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for body, name in re.findall(r"typedef struct\s*\{(.*?)\}\s*(\w+)\s*;", text, flags=re.S):
        names = []
        for decl in body.split(";"):
            decl = decl.strip()
            if not decl:
                continue
            parts = [p.strip() for p in decl.split(",")]
            names.append(re.split(r"[\s*]+", parts[0])[-1])
            names.extend(p.strip("* ") for p in parts[1:])
        out[name] = names
    return out


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    fields = _header_fields()
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "lnfp8.h"', "int main(void) {"]
    for s in STRUCTS:
        lines.append(f'  printf("{s} size %zu\\n", sizeof({s}));')
        for f in fields[s]:
            lines.append(f'  printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    res = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        s, f, v = line.split()
        res[(s, f)] = int(v)
    return fields, res


@pytest.mark.parametrize("cname", sorted(STRUCTS))
def test_ctypes_struct_matches_header(c_layout, cname):
    import importlib.util
    spec = importlib.util.find_spec("fp8_delayed_scaling_row_gb300.lnfp8")
    if spec is None:
        pytest.skip("binding not importable")
    try:
        from fp8_delayed_scaling_row_gb300 import lnfp8
    except OSError as e:  # library not built
        pytest.skip(str(e))
    fields, res = c_layout
    cls = getattr(lnfp8, STRUCTS[cname])
    assert [f[0] for f in cls._fields_] == fields[cname]
    assert ctypes.sizeof(cls) == res[(cname, "size")]
    for f in fields[cname]:
        assert getattr(cls, f).offset == res[(cname, f)], f
