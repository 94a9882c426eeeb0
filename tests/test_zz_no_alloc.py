"""fp8_quantize_static_scratch against fp8_quantize, through the C ABI.

The allocation-free entry point serves callers that cannot give the library device memory
(a host framework whose allocator owns the whole pool, or loops that must not pay for
cudaMalloc's implicit synchronisation). It must produce exactly what the workspace-taking
entry point produces, on two calls in a row (the second call reuses the shared array that the
first one left behind). This file sorts last so a run that stops at the first failure has
already run every other test; it also passes when run alone in a fresh process.
"""
import ctypes
import os
import subprocess
import sys

import pytest
import torch

from helpers import cuda_ok, same_f32, to_dev_bf16
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import _lib as L


@pytest.mark.parametrize("kind", ["tensorwise", "delayed", "mxfp8"])
def test_static_scratch_matches_workspace_entry(kind):
    rec = F.Recipe(kind=kind, amax_history_len=16)
    shapes = [(1024, 768), (272, 4096)] if kind != "mxfp8" else [(1024, 768), (384, 4096)]
    for call, (R, C) in enumerate(shapes):           # two calls in a row, different sizes
        x = to_dev_bf16(bf16_bits_normal(R, C, seed=70 + call, sigma=3.0))
        ref = F.empty_qtensor(rec, R, C)
        got = F.empty_qtensor(rec, R, C)
        if kind == "delayed":
            for q in (ref, got):
                q.scale.fill_(448.0 / 7.0)
                q.scale_inv.fill_(7.0 / 448.0)
        F.quantize(rec, x, out=ref)
        F.quantize_static_scratch(rec, x, out=got)
        torch.cuda.synchronize()
        assert torch.equal(got.row, ref.row) and torch.equal(got.col, ref.col)
        if kind == "mxfp8":
            assert torch.equal(got.row_scale, ref.row_scale)
            assert torch.equal(got.col_scale, ref.col_scale)
        else:
            assert same_f32(got.amax.item(), ref.amax.item())
            assert same_f32(got.scale.item(), ref.scale.item())
            assert same_f32(got.scale_inv.item(), ref.scale_inv.item())


def test_static_scratch_rejects_oversized():
    """More 128 x 128 tiles than the array has partial slots: rejected before any launch."""
    lib = L.load()
    rc = F.Recipe(kind="delayed").c()
    x = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    q = F.empty_qtensor(F.Recipe(kind="delayed"), 16, 16)
    t = q.c()
    st = lib.fp8_quantize_static_scratch(ctypes.byref(rc), ctypes.c_void_p(x.data_ptr()),
                                         128 * 65537, 128, 0, 1, 1, ctypes.byref(t), None, None)
    assert st == 7                                   # FP8_ERR_WORKSPACE


def test_static_scratch_after_device_reset():
    """A cudaDeviceReset gives the device a new context, in which the scratch array may sit at
    another address: the entry point must look it up again rather than reuse the old one (and
    the kernels' shared-memory attributes must be set again). Run in a child process without
    torch, whose allocator would otherwise hold pointers the reset invalidates; the child
    compares the entry point with fp8_quantize before and after the reset."""
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "noalloc_reset_child.py")
    r = subprocess.run([sys.executable, child], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.returncode, r.stdout[-2000:], r.stderr[-2000:])
