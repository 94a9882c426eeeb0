"""The binding's ctypes prototypes match the C declarations in include/*.h: every declared
function has a prototype, with the same number of arguments and the same kind of each (a
pointer, a 32- or 64-bit integer, a size). A mismatch would pass garbage at call time, which
on a CPU-only machine nothing else would notice."""
import ctypes
import os
import re

import pytest

from scaled_quantize_fp8_gb300 import _lib as L

DECL = re.compile(r"^\s*(?:fp8_status|size_t|const char \*)\s*(fp8_\w+)\s*\(([^;]*?)\)\s*;",
                  re.M | re.S)


def declarations():
    out = {}
    for h in sorted(os.listdir(L.HEADER_DIR)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(L.HEADER_DIR, h)).read(), flags=re.S)
            for name, params in DECL.findall(text):
                out[name] = [p.strip() for p in params.split(",")] if params.strip() != "void" else []
    return out


def c_kind(param):
    """'ptr', 'i32', 'i64' or 'size' for one C parameter declaration."""
    t = re.sub(r"\b\w+\s*$", "", param) if "*" not in param.split()[-1] else param
    if "*" in param or "cudaStream_t" in param:
        return "ptr"
    if "int64_t" in t:
        return "i64"
    if "size_t" in t:
        return "size"
    if "int32_t" in t or "fp8_status" in t or re.search(r"\bint\b", t):
        return "i32"
    raise AssertionError(f"unclassified C parameter: {param!r}")


def ctypes_kind(ct):
    if ct in (ctypes.c_void_p, ctypes.c_char_p) or isinstance(ct, type(ctypes.POINTER(ctypes.c_int))):
        return "ptr"
    if ct is ctypes.c_int32:
        return "i32"
    if ct is ctypes.c_int64:
        return "i64"
    if ct is ctypes.c_size_t:
        return "size"
    raise AssertionError(f"unclassified ctypes type: {ct!r}")


DECLS = declarations()


def test_every_declared_function_has_a_prototype():
    assert set(DECLS) == set(L.header_functions())
    missing = sorted(set(DECLS) - set(L._SIG))
    assert missing == [], missing


@pytest.mark.parametrize("name", sorted(DECLS))
def test_prototype_matches_declaration(name):
    want = [c_kind(p) for p in DECLS[name]]
    got = [ctypes_kind(t) for t in L._SIG[name][1]]
    assert got == want, (name, DECLS[name])


def test_parser_sees_a_mismatch():
    """The comparison itself: a prototype with one argument too few is reported."""
    params = ["const fp8_recipe *recipe", "int64_t rows", "int64_t cols"]
    assert [c_kind(p) for p in params] == ["ptr", "i64", "i64"]
    assert [ctypes_kind(t) for t in [ctypes.c_void_p, ctypes.c_int64]] != \
        [c_kind(p) for p in params]
