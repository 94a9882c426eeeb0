"""Shared helpers for the parity tests: device transfer, scale-layout index maps, tolerances.

Nothing here computes any part of the FP8 method; it moves bytes and compares results.
"""
import numpy as np
import torch

# Tolerances: elementwise relative error of bf16 GEMM outputs with a floor at 1e-3 of the
# output's max magnitude (rounding to bf16 alone contributes up to 2^-9), and the normwise
# error of the fp32-output mode against the fp64 reference on the same FP8 operands.
GEMM_BF16_RTOL = 1e-2
GEMM_F32_NORMWISE = 1e-5


def cuda_ok():
    return torch.cuda.is_available()


def to_dev_bf16(bits):
    """numpy uint16 bf16 patterns -> torch bf16 tensor on the GPU."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def from_dev_bf16(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def mx_untile(tiled, rows, cols):
    """Tiled E8M0 bytes of a [rows][cols] copy -> plain [rows][cols/32] (index map only)."""
    r = np.arange(rows)[:, None]
    kb = np.arange(cols // 32)[None, :]
    off = ((r >> 7) * (cols >> 7) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (kb & 3)
    return np.asarray(tiled).reshape(-1)[off]


def bw_untile(blockmajor, rows, cols):
    """1x128 s_inv stored [cols/128][rows] -> [rows][cols/128]."""
    return np.ascontiguousarray(np.asarray(blockmajor).reshape(cols // 128, rows).T)


def gemm_bf16_close(got_bits, ref64, rtol=GEMM_BF16_RTOL):
    """Elementwise |C - R| / max(|R|, 1e-3 max|R|) <= rtol; returns the worst ratio."""
    from oracle.fp8_oracle import bf16_to_f32
    c = bf16_to_f32(got_bits).astype(np.float64)
    floor = 1e-3 * np.max(np.abs(ref64)) if ref64.size else 0.0
    den = np.maximum(np.abs(ref64), floor)
    den = np.where(den == 0, 1.0, den)
    worst = float(np.max(np.abs(c - ref64) / den)) if ref64.size else 0.0
    return worst <= rtol, worst


def gemm_f32_normwise(got_f32, ref64):
    if ref64.size == 0:
        return True, 0.0
    m = np.max(np.abs(ref64))
    err = float(np.max(np.abs(got_f32.astype(np.float64) - ref64)) / (m if m > 0 else 1.0))
    return err <= GEMM_F32_NORMWISE, err


def same_f32(a, b):
    """Bit-identical float32 scalars, or both NaN (a NaN's payload is not part of the result)."""
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a.tobytes() == b.tobytes()
