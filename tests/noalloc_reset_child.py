"""Child process of test_zz_no_alloc: fp8_quantize_static_scratch across a cudaDeviceReset.

The allocation-free entry point looks up its scratch array's device address once per CUDA
context. A reset destroys the device's primary context; the next CUDA call makes a new one, in
which the library's device image, and so the array, may sit at another address. This process
runs the entry point before and after a reset and compares it, byte for byte, with
fp8_quantize given a workspace, for the tensorwise and delayed recipes (the two that use the
scratch array), plus an MXFP8 quantize (whose kernel needs its shared-memory attribute set
again in the new context).

It loads no torch, so the only CUDA runtime in the process is the one the library links, and
the reset cannot leave another runtime holding dead pointers. Buffers come from cudaMalloc
through ctypes. Before the post-reset call it checks that the context id did change, and
exits with status 3 without calling the entry point if it did not. Exit status 0 means every
comparison held.
"""
import ctypes
import importlib.util
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location(
    "fp8lin_abi", os.path.join(ROOT, "scaled_quantize_fp8_gb300", "_lib.py"))
L = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(L)

lib = L.load()
_cudart_path = next(ln.split()[-1] for ln in open("/proc/self/maps") if "libcudart" in ln)
rt = ctypes.CDLL(_cudart_path)
drv = ctypes.CDLL("libcuda.so.1")
H2D, D2H = 1, 2


def ok(e, what):
    if e != 0:
        raise RuntimeError(f"{what} failed with CUDA error {e}")


def dmalloc(n):
    p = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(n, 16))), "cudaMalloc")
    return p.value


def h2d(dst, arr):
    arr = np.ascontiguousarray(arr)
    ok(rt.cudaMemcpy(ctypes.c_void_p(dst), arr.ctypes.data_as(ctypes.c_void_p),
                     ctypes.c_size_t(arr.nbytes), H2D), "cudaMemcpy H2D")


def d2h(src, nbytes):
    out = np.empty(nbytes, np.uint8)
    ok(rt.cudaMemcpy(out.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(src),
                     ctypes.c_size_t(nbytes), D2H), "cudaMemcpy D2H")
    return out


def context_id():
    ctx = ctypes.c_void_p()
    ok(drv.cuCtxGetCurrent(ctypes.byref(ctx)), "cuCtxGetCurrent")
    if not ctx.value:
        return 0
    cid = ctypes.c_ulonglong()
    ok(drv.cuCtxGetId(ctx, ctypes.byref(cid)), "cuCtxGetId")
    return cid.value


def bf16_bits(R, C, seed):
    """Arbitrary finite bf16 patterns (the top halves of normal float32 samples)."""
    f = (np.random.default_rng(seed).standard_normal((R, C)) * 3.0).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def quantized(kind, x_dev, R, C, static, ws=None):
    """One quantize into fresh buffers; returns the bytes of every output."""
    row, col = dmalloc(R * C), dmalloc(R * C)
    rs = cs = None
    if kind == L.RECIPE_MXFP8:
        rs, cs = dmalloc(R * C // 32), dmalloc(R * C // 32)
    amax, scale, sinv = dmalloc(4), dmalloc(4), dmalloc(4)
    if kind == L.RECIPE_DELAYED:                 # the scale an earlier history produced
        h2d(scale, np.array([448.0 / 7.0], np.float32))
        h2d(sinv, np.array([7.0 / 448.0], np.float32))
    t = L.Tensor(row, col, rs, cs, amax, scale, sinv, 0, 0, 0, 0, 0)
    rec = L.Recipe(kind, L.FORMAT_E4M3, 0, 16, 0, 1, 0)
    if static:
        st = lib.fp8_quantize_static_scratch(ctypes.byref(rec), ctypes.c_void_p(x_dev), R, C,
                                             L.ROLE_ACTIVATION, 1, 1, ctypes.byref(t), None,
                                             None)
    else:
        st = lib.fp8_quantize(ctypes.byref(rec), ctypes.c_void_p(x_dev), R, C,
                              L.ROLE_ACTIVATION, 1, 1, ctypes.byref(t), ctypes.c_void_p(ws[0]),
                              ws[1], None, None)
    if st != 0:
        raise RuntimeError(f"quantize returned {L.STATUS_NAMES.get(st, st)}: "
                           f"{lib.fp8_last_cuda_error().decode()}")
    ok(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
    out = {"row": d2h(row, R * C), "col": d2h(col, R * C), "amax": d2h(amax, 4),
           "scale": d2h(scale, 4), "scale_inv": d2h(sinv, 4)}
    if rs is not None:
        out["row_scale"], out["col_scale"] = d2h(rs, R * C // 32), d2h(cs, R * C // 32)
    return out


def one_round(seed):
    R, C = 1024, 768
    x = dmalloc(R * C * 2)
    h2d(x, bf16_bits(R, C, seed))
    for kind in (L.RECIPE_TENSORWISE, L.RECIPE_DELAYED, L.RECIPE_MXFP8):
        rec = L.Recipe(kind, L.FORMAT_E4M3, 0, 16, 0, 1, 0)
        need = lib.fp8_workspace_bytes(ctypes.byref(rec), R, C)
        ws = (dmalloc(need), need) if need else (None, 0)
        ref = quantized(kind, x, R, C, static=False, ws=ws)
        got = quantized(kind, x, R, C, static=True)
        for name in ref:
            if not np.array_equal(ref[name], got[name]):
                raise AssertionError(f"kind {kind}: {name} differs (seed {seed})")


def main():
    ok(rt.cudaSetDevice(0), "cudaSetDevice")
    one_round(seed=1)
    before = context_id()
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    dmalloc(16)                                    # the runtime makes its new context here
    after = context_id()
    if before == 0 or after == before:
        print(f"context id did not change across the reset ({before} -> {after})")
        return 3
    one_round(seed=2)
    print(f"ok: context {before} -> {after}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
