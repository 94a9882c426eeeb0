"""The binding's ctypes structures have the C structs' layout: a small C program compiled
against include/fp8lin.h prints sizeof and every field's offset of fp8_recipe, fp8_tensor,
fp8_amax_history and fp8_quantize_item, and the ctypes Structure classes must agree field by
field."""
import ctypes
import os
import shutil
import subprocess

import pytest

from scaled_quantize_fp8_gb300 import _lib as L

STRUCTS = {"fp8_recipe": L.Recipe, "fp8_tensor": L.Tensor, "fp8_amax_history": L.AmaxHistory,
           "fp8_quantize_item": L.QuantizeItem}


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    return None


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if cc is None or inc is None:
        pytest.skip("needs a C compiler and the CUDA runtime headers")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fp8lin.h"', 'int main(void) {']
    for cname, cls in STRUCTS.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("layout")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    r = subprocess.run([cc, "-std=c99", "-I", L.HEADER_DIR, "-I", inc, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    table = {}
    for line in out.splitlines():
        name, field, value = line.split()
        table[(name, field)] = int(value)
    return table


@pytest.mark.parametrize("cname", sorted(STRUCTS))
def test_struct_layout_matches(c_layout, cname):
    cls = STRUCTS[cname]
    assert ctypes.sizeof(cls) == c_layout[(cname, "size")]
    for fname, _ in cls._fields_:
        assert getattr(cls, fname).offset == c_layout[(cname, fname)], fname
