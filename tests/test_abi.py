"""C ABI checks that need no GPU: the library loads, exports every function the header
declares, and rejects bad arguments on the host before launching anything."""
import ctypes

import pytest
import torch

from scaled_quantize_fp8_gb300 import _lib as L
from scaled_quantize_fp8_gb300 import build as B


# These tests hand the library made-up device addresses that host-side validation must reject
# before anything is launched. They never run where a GPU is visible, so a validation gap can
# never turn into a kernel touching those addresses.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake-pointer validation tests run on CPU-only hosts")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def _rec(kind=L.RECIPE_TENSORWISE, fmt=L.FORMAT_E4M3, margin=0, hist=16, algo=0, wgrad=1):
    return L.Recipe(kind, fmt, margin, hist, algo, wgrad)


def _tensor(row=0x1000, col=0x2000, rs=0x3000, cs=0x4000, amax=0x5000, scale=0x6000,
            sinv=0x7000):
    return L.Tensor(row, col, rs, cs, amax, scale, sinv, 0, 0, 0, 0, 0)


def test_exports_every_declared_symbol(lib):
    names = L.header_functions()
    assert {"fp8_quantize", "fp8_amax_update", "fp8_linear_fwd", "fp8_linear_bwd"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        assert lib.fp8_status_str(code)
    assert lib.fp8_last_cuda_error() == b""


def _q(lib, rec, x=0x8000, rows=256, cols=256, role=0, wr=1, wc=1, t=None, ws=0x9000,
       ws_bytes=1 << 20):
    t = t or _tensor()
    return lib.fp8_quantize(ctypes.byref(rec), x, rows, cols, role, wr, wc, ctypes.byref(t), ws,
                            ws_bytes, None, None)


def _group(lib, rec, items, n=None):
    arr = (L.QuantizeItem * max(1, len(items)))(*items)
    return lib.fp8_quantize_group(ctypes.byref(rec), len(items) if n is None else n, arr, None,
                                  None)


def _item(t, x=0x8000, rows=256, cols=256, role=0, wr=1, wc=1):
    return L.QuantizeItem(x, rows, cols, role, wr, wc, ctypes.pointer(t))


def test_quantize_group_rejects_bad_arguments(lib):
    mx = _rec(kind=L.RECIPE_MXFP8)
    t0, t1 = _tensor(), _tensor(row=0x11000, col=0x12000, rs=0x13000, cs=0x14000)
    assert lib.fp8_quantize_group(None, 1, None, None, None) == 1
    assert _group(lib, _rec(), [_item(t0)]) == 4                 # MXFP8 and blockwise only
    assert _group(lib, _rec(kind=L.RECIPE_DELAYED), [_item(t0)]) == 4
    assert _group(lib, _rec(kind=L.RECIPE_BLOCKWISE), [_item(t0, cols=64)]) == 3
    assert _group(lib, _rec(kind=L.RECIPE_MXFP8, fmt=L.FORMAT_HYBRID), [_item(t0)]) == 4
    assert lib.fp8_quantize_group(ctypes.byref(mx), 1, None, None, None) == 1
    assert _group(lib, mx, [_item(t0)], n=0) == 3
    assert _group(lib, mx, [_item(t0)] * 5) == 3               # at most FP8_QUANTIZE_GROUP_MAX
    assert _group(lib, mx, [_item(t0), _item(t1, rows=192)]) == 3    # item 1: not a 128 multiple
    assert _group(lib, mx, [_item(t0), _item(t1, x=0)]) == 1
    assert _group(lib, mx, [_item(t0, x=0x8008), _item(t1)]) == 2
    assert _group(lib, mx, [_item(t0), _item(t1, role=7)]) == 4
    assert _group(lib, mx, [_item(t0), _item(t1, wr=0, wc=0)]) == 3
    assert _group(lib, mx, [_item(t0), _item(_tensor(rs=0))]) == 1
    bad = L.QuantizeItem(0x8000, 256, 256, 0, 1, 1, None)     # no output tensor
    assert _group(lib, mx, [_item(t0), bad]) == 1
    # nothing launched and no output touched when any item fails
    assert t0.rows == 0 and t0.cols == 0 and t0.kind == 0


def test_quantize_rejects_bad_arguments(lib):
    r = _rec()
    assert lib.fp8_quantize(None, 0x8000, 16, 16, 0, 1, 1, ctypes.byref(_tensor()), None, 0, None,
                            None) == 1
    assert _q(lib, _rec(kind=L.RECIPE_MXFP8, fmt=L.FORMAT_HYBRID)) == 4   # mxfp8: E4M3 only
    assert _q(lib, _rec(fmt=3)) == 4                           # no such format
    assert _q(lib, _rec(kind=9)) == 4
    assert _q(lib, _rec(margin=65)) == 4
    assert _q(lib, _rec(algo=2)) == 4                          # max or most_recent
    pow2 = _rec()
    pow2.power_2_scales = 1
    assert _q(lib, pow2) == 4                                  # power-of-two: blockwise only
    assert _q(lib, _rec(kind=L.RECIPE_DELAYED, hist=0)) == 3
    assert _q(lib, r, rows=-16) == 3
    assert _q(lib, r, rows=24) == 3                            # not a multiple of 16
    assert _q(lib, _rec(kind=L.RECIPE_MXFP8), rows=192, cols=160) == 3   # MX needs 128
    assert _q(lib, _rec(kind=L.RECIPE_BLOCKWISE), cols=64) == 3
    assert _q(lib, r, wr=0, wc=0) == 3
    assert _q(lib, r, x=0) == 1
    assert _q(lib, r, x=0x8008) == 2                           # misaligned input
    assert _q(lib, r, t=_tensor(row=0)) == 1
    assert _q(lib, r, t=_tensor(col=0x2001)) == 2
    assert _q(lib, r, t=_tensor(amax=0)) == 1
    assert _q(lib, _rec(kind=L.RECIPE_MXFP8), t=_tensor(rs=0)) == 1
    assert _q(lib, _rec(kind=L.RECIPE_BLOCKWISE), t=_tensor(cs=0x4004)) == 2
    assert _q(lib, r, role=7) == 4


def test_quantize_workspace_checks(lib):
    r = _rec(kind=L.RECIPE_DELAYED)
    need = lib.fp8_workspace_bytes(ctypes.byref(r), 256, 256)
    assert need == 4 * 4                                       # one partial per 128x128 tile
    assert _q(lib, r, ws=0) == 7
    assert _q(lib, r, ws_bytes=need - 1) == 7
    assert _q(lib, r, ws=0x9004) == 2
    assert lib.fp8_workspace_bytes(ctypes.byref(_rec(kind=L.RECIPE_MXFP8)), 256, 256) == 0


def test_amax_update_checks(lib):
    r = _rec(kind=L.RECIPE_DELAYED, hist=8)
    h = L.AmaxHistory(0x1000, 0x2000, 8)
    assert lib.fp8_amax_update(ctypes.byref(_rec(kind=L.RECIPE_MXFP8)), ctypes.byref(h), 0,
                               0x3000, 0x4000, 0x5000, None) == 4
    bad = L.AmaxHistory(0x1000, 0x2000, 4)                    # length differs from the recipe
    assert lib.fp8_amax_update(ctypes.byref(r), ctypes.byref(bad), 0, 0x3000, 0x4000, 0x5000,
                               None) == 3
    assert lib.fp8_amax_update(ctypes.byref(r), ctypes.byref(h), 0, None, 0x4000, 0x5000,
                               None) == 1
    assert lib.fp8_amax_update(ctypes.byref(r), ctypes.byref(h), 5, 0x3000, 0x4000, 0x5000,
                               None) == 4                      # no such role


def _qt(kind, rows, cols, role=0):
    t = _tensor()
    t.rows, t.cols, t.kind, t.role = rows, cols, kind, role
    return t


def test_linear_fwd_checks(lib):
    r = _rec(kind=L.RECIPE_MXFP8)
    x, w = _qt(L.RECIPE_MXFP8, 256, 512), _qt(L.RECIPE_MXFP8, 384, 512, 1)
    fwd = lib.fp8_linear_fwd
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(_qt(L.RECIPE_MXFP8, 384, 256)),
               0x1000, 0, None, None) == 3                    # K mismatch
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(_qt(L.RECIPE_TENSORWISE, 384, 512)),
               0x1000, 0, None, None) == 4                    # recipes differ
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), 0, 0, None, None) == 1
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), 0x1008, 0, None, None) == 2
    xr = _qt(L.RECIPE_MXFP8, 200, 512)
    assert fwd(ctypes.byref(r), ctypes.byref(xr), ctypes.byref(w), 0x1000, 0, None, None) == 3
    rb = _rec(kind=L.RECIPE_BLOCKWISE)
    xa = _qt(L.RECIPE_BLOCKWISE, 256, 512, 1)                 # A must be 1x128, not a weight
    wb = _qt(L.RECIPE_BLOCKWISE, 384, 512, 1)
    assert fwd(ctypes.byref(rb), ctypes.byref(xa), ctypes.byref(wb), 0x1000, 0, None, None) == 4


def test_stalled_fwd_hook_checks(lib):
    """The failure-detection hook validates like fp8_linear_fwd and needs a status word."""
    r = _rec(kind=L.RECIPE_MXFP8)
    x, w = _qt(L.RECIPE_MXFP8, 256, 512), _qt(L.RECIPE_MXFP8, 384, 512, 1)
    hook = lib.fp8_test_linear_fwd_stalled
    assert hook(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), 0x1000, None, None) == 1
    assert hook(ctypes.byref(r), ctypes.byref(x), ctypes.byref(_qt(L.RECIPE_MXFP8, 384, 256)),
                0x1000, 0x9000, None) == 3                   # K mismatch
    assert hook(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), 0, 0x9000, None) == 1


def test_stalled_quantize_hook_checks(lib):
    """The quantize hook validates like fp8_quantize and needs a status word."""
    r = _rec(kind=L.RECIPE_MXFP8)
    out = _tensor()
    hook = lib.fp8_test_quantize_stalled
    assert hook(ctypes.byref(r), 0x1000, 256, 256, 0, 1, 1, ctypes.byref(out), None, 0, None,
                None) == 1
    assert hook(ctypes.byref(r), 0x1000, 200, 256, 0, 1, 1, ctypes.byref(out), None, 0, 0x9000,
                None) == 3                                     # rows not a multiple of 128


def test_linear_bwd_checks(lib):
    r = _rec(kind=L.RECIPE_TENSORWISE)
    dy = _qt(L.RECIPE_TENSORWISE, 256, 384)
    x = _qt(L.RECIPE_TENSORWISE, 256, 512)
    w = _qt(L.RECIPE_TENSORWISE, 384, 512)
    bwd = lib.fp8_linear_bwd
    assert bwd(ctypes.byref(r), ctypes.byref(dy), ctypes.byref(x),
               ctypes.byref(_qt(L.RECIPE_TENSORWISE, 320, 512)), 0x1000, None, 0,
               None, None) == 3                               # W rows != dY cols
    assert bwd(ctypes.byref(r), ctypes.byref(dy), ctypes.byref(_qt(L.RECIPE_TENSORWISE, 128, 512)),
               ctypes.byref(w), None, 0x1000, 0, None, None) == 3
    assert bwd(ctypes.byref(r), None, ctypes.byref(x), ctypes.byref(w), 0x1000,
               0x2000, 0, None, None) == 1
    # --fp8-wgrad off needs column copies made under that recipe (bf16 transposes)
    r_off = _rec(kind=L.RECIPE_TENSORWISE, wgrad=0)
    assert bwd(ctypes.byref(r_off), ctypes.byref(dy), ctypes.byref(x), ctypes.byref(w), None,
               0x1000, 0, None, None) == 4


def test_mlp_entry_checks(lib):
    r = _rec(kind=L.RECIPE_MXFP8)
    a, h = _tensor(), _tensor()
    assert lib.fp8_gelu_quantize(ctypes.byref(_rec()), 0x1000, 256, 256, None, ctypes.byref(a),
                                 ctypes.byref(h), None, None) == 4
    assert lib.fp8_gelu_quantize(ctypes.byref(r), 0x1000, 256, 200, None, ctypes.byref(a),
                                 ctypes.byref(h), None, None) == 3
    assert lib.fp8_gelu_quantize(ctypes.byref(r), 0x1000, 256, 256, 0x2008, ctypes.byref(a),
                                 ctypes.byref(h), None, None) == 2
    hq = _qt(L.RECIPE_TENSORWISE, 256, 256)
    assert lib.fp8_dgelu_quantize(ctypes.byref(r), 0x1000, ctypes.byref(hq), None,
                                  ctypes.byref(_tensor()), None, None) == 4


def test_fused_mlp_entry_checks(lib):
    r = _rec(kind=L.RECIPE_MXFP8)
    x, w = _qt(L.RECIPE_MXFP8, 256, 512), _qt(L.RECIPE_MXFP8, 384, 512, 1)
    a, h = _tensor(), _tensor()
    fwd = lib.fp8_linear_fwd_gelu
    assert fwd(ctypes.byref(_rec()), ctypes.byref(x), ctypes.byref(w), ctypes.byref(a),
               ctypes.byref(h), None, None) == 4                 # MXFP8 only
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(_qt(L.RECIPE_MXFP8, 384, 256, 1)),
               ctypes.byref(a), ctypes.byref(h), None, None) == 3   # K mismatch
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(h), None,
               None) == 1
    assert fwd(ctypes.byref(r), ctypes.byref(_qt(L.RECIPE_MXFP8, 200, 512)), ctypes.byref(w),
               ctypes.byref(a), ctypes.byref(h), None, None) == 3   # M not a multiple of 128
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), ctypes.byref(a),
               ctypes.byref(_tensor(row=0x1008)), None, None) == 2  # misaligned h codes
    assert fwd(ctypes.byref(r), ctypes.byref(x), ctypes.byref(w), ctypes.byref(_tensor(cs=0)),
               ctypes.byref(h), None, None) == 1
    dgr = lib.fp8_linear_dgrad_dgelu
    dy, w2 = _qt(L.RECIPE_MXFP8, 256, 384), _qt(L.RECIPE_MXFP8, 384, 512, 1)
    hq = _qt(L.RECIPE_MXFP8, 256, 512)
    assert dgr(ctypes.byref(r), ctypes.byref(dy), ctypes.byref(w2),
               ctypes.byref(_qt(L.RECIPE_MXFP8, 256, 384)), ctypes.byref(_tensor()), None,
               None) == 3                                        # h is [M][w2 cols]
    assert dgr(ctypes.byref(r), ctypes.byref(dy), ctypes.byref(w2),
               ctypes.byref(_qt(L.RECIPE_TENSORWISE, 256, 512)), ctypes.byref(_tensor()), None,
               None) == 4
    assert dgr(ctypes.byref(r), ctypes.byref(dy), ctypes.byref(w2), ctypes.byref(hq), None,
               None, None) == 1
