"""Backward GEMMs that read a row-wise copy as an MN-major (transposed) tensor-core operand, for
tensors quantised without their column copy: per-tensor recipes (dgrad's W, wgrad's dY and X)
and blockwise 128x128 weights (dgrad's W). Checked against the oracle and against the same
GEMMs on the column copies."""
import numpy as np
import pytest
import torch

from helpers import (cuda_ok, from_dev_bf16, gemm_bf16_close, gemm_f32_normwise, to_dev_bf16)
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _quant(rec, b, role, want_col, scale=None):
    q = F.empty_qtensor(rec, b.shape[0], b.shape[1], role, True, want_col)
    if scale is not None:
        q.scale.fill_(float(scale[0]))
        q.scale_inv.fill_(float(scale[1]))
    return F.quantize(rec, to_dev_bf16(b), role, True, want_col, out=q)


def _oracle_pair(kind, b, role, fmt, scale):
    """(row deq, col deq) of the oracle's quantisation of b."""
    if kind == "tensorwise":
        q = O.quantize_tensorwise(b, fmt=fmt)
    elif kind == "delayed":
        d = O.DelayedScaling(4, fmt=fmt)
        d.scale, d.scale_inv = scale
        q = d.quantize(b)
    if kind in ("tensorwise", "delayed"):
        return (O.dequant_tensor(q["row"], q["scale_inv"], fmt),
                O.dequant_tensor(q["col"], q["scale_inv"], fmt))
    if role == "weight":
        q = O.quantize_blockwise_128x128(b, fmt=fmt)
        return (O.dequant_128x128(q["row"], q["row_scale_inv"], fmt),
                O.dequant_128x128(q["col"], q["col_scale_inv"], fmt))
    q = O.quantize_blockwise_1x128(b, fmt=fmt)
    return (O.dequant_1x128(q["row"], q["row_scale_inv"], fmt),
            O.dequant_1x128(q["col"], q["col_scale_inv"], fmt))


@pytest.mark.parametrize("kind,fmt", [("tensorwise", "e4m3"), ("delayed", "e4m3"),
                                      ("tensorwise", "hybrid"), ("blockwise", "e4m3")])
# the last two shapes give dgrad (dX 2560 x 4096) and wgrad (dW 4096 x 2560), each reading
# MN-major operands, more tiles than the grid runs at once
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (128, 256, 384), (384, 256, 128),
                                   (2560, 256, 4096), (256, 4096, 2560)])
@pytest.mark.parametrize("fp32", [False, True])
def test_bwd_without_column_copies(kind, fmt, M, N, K, fp32):
    rec = F.Recipe(kind=kind, format=fmt)
    xb = bf16_bits_normal(M, K, seed=M + K)
    wb = bf16_bits_normal(N, K, seed=N + K, sigma=0.02)
    dyb = bf16_bits_normal(M, N, seed=M + N, sigma=1e-3)
    per_tensor = kind != "blockwise"
    q_mn, q_col, ref = {}, {}, {}
    for name, b, role in (("x", xb, "activation"), ("w", wb, "weight"), ("dy", dyb, "grad")):
        f = O.hybrid_format(role) if fmt == "hybrid" else "e4m3"
        sc = None
        if kind == "delayed":
            sc = O.scale_from_amax(O.amax_of(b) * np.float32(1.25), 0, f)
        # the column copy is dropped wherever the row copy can stand in for it
        drop = per_tensor or role == "weight"
        q_mn[name] = _quant(rec, b, role, not drop, sc)
        q_col[name] = _quant(rec, b, role, True, sc)
        ref[name] = _oracle_pair(kind, b, role, f, sc)
    assert q_mn["w"].col is None and (not per_tensor or q_mn["dy"].col is None)
    dx, dw = F.linear_bwd(rec, q_mn["dy"], q_mn["x"], q_mn["w"], fp32=fp32)
    dx_c, dw_c = F.linear_bwd(rec, q_col["dy"], q_col["x"], q_col["w"], fp32=fp32)
    torch.cuda.synchronize()
    dx_ref = O.gemm_tn_f64(ref["dy"][0], ref["w"][1])
    dw_ref = O.gemm_tn_f64(ref["dy"][1], ref["x"][1])
    for got, ref_, other in ((dx, dx_ref, dx_c), (dw, dw_ref, dw_c)):
        if fp32:
            ok, err = gemm_f32_normwise(got.cpu().numpy(), ref_)
            assert ok, err
            assert np.max(np.abs(got.cpu().numpy() - other.cpu().numpy())) <= \
                1e-6 * np.max(np.abs(ref_))
        else:
            ok, err = gemm_bf16_close(from_dev_bf16(got), ref_)
            assert ok, err
