"""GPU parity of the hybrid format (--fp8-format hybrid): gradients stored in E5M2, activations
and weights in E4M3, for the delayed, tensorwise and blockwise recipes, and the mixed
E5M2 x E4M3 dgrad / wgrad GEMMs. Codes and scales are bit-exact against the oracle; GEMMs are
graded like the E4M3 ones (elementwise 1e-2 on bf16 outputs, normwise 1e-5 in fp32 mode).
"""
import numpy as np
import pytest
import torch

from helpers import (bw_untile, cuda_ok, from_dev_bf16, gemm_bf16_close, gemm_f32_normwise,
                     mx_untile, same_f32, to_dev_bf16)
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _np(t):
    return t.cpu().numpy()


def _q(kind, x_bits, role, margin=0, scale=None):
    rec = F.Recipe(kind=kind, format="hybrid", margin=margin)
    out = F.empty_qtensor(rec, x_bits.shape[0], x_bits.shape[1], role)
    if scale is not None:
        out.scale.fill_(float(scale))
        out.scale_inv.fill_(float(np.float32(1.0) / np.float32(scale)))
    F.quantize(rec, to_dev_bf16(x_bits), role, out=out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("role", ["grad", "activation", "weight"])
@pytest.mark.parametrize("margin", [0, 2])
def test_tensorwise_hybrid(role, margin):
    x = bf16_bits_normal(256, 384, seed=71, sigma=1e-3 if role == "grad" else 1.0)
    q = _q("tensorwise", x, role, margin)
    ref = O.quantize_tensorwise(x, margin, fmt=O.hybrid_format(role))
    assert same_f32(_np(q.scale)[0], ref["scale"])
    assert same_f32(_np(q.scale_inv)[0], ref["scale_inv"])
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


@pytest.mark.parametrize("role", ["grad", "weight"])
def test_blockwise_hybrid(role):
    x = bf16_bits_normal(256, 384, seed=72, sigma=1e-3, outlier_p=1e-2, outlier_factor=30.0)
    R, C = x.shape
    q = _q("blockwise", x, role)
    fmt = O.hybrid_format(role)
    if role == "weight":
        ref = O.quantize_blockwise_128x128(x, fmt=fmt)
        assert np.array_equal(_np(q.row_scale), ref["row_scale_inv"])
    else:
        ref = O.quantize_blockwise_1x128(x, fmt=fmt)
        assert np.array_equal(bw_untile(_np(q.row_scale), R, C), ref["row_scale_inv"])
        assert np.array_equal(bw_untile(_np(q.col_scale), C, R), ref["col_scale_inv"])
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


@pytest.mark.parametrize("scale", [1.0, 3.0, 2.0 ** -14, 2.0 ** 10, 1e-30, 1e30])
def test_exhaustive_bf16_e5m2_cast(scale):
    """Every bf16 bit pattern (zeros, subnormals, the largest values, Inf, NaN) cast to E5M2
    with a fixed delayed scale: the hardware conversion against the oracle's reading."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    q = _q("delayed", x, "grad", scale=scale)
    d = O.DelayedScaling(4, fmt="e5m2")
    d.scale = np.float32(scale)
    ref = d.quantize(x)
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


def test_delayed_hybrid_history():
    """A gradient's delayed history under hybrid derives its scale from 57344."""
    rec = F.Recipe(kind="delayed", format="hybrid", amax_history_len=4)
    state = F.DelayedState(rec, role="grad")
    d = O.DelayedScaling(4, fmt="e5m2")
    for t, sigma in enumerate([1e-3, 4e-3, 2e-4, 1e-2, 5e-4, 3e-3]):
        x = bf16_bits_normal(128, 256, seed=80 + t, sigma=sigma)
        q = F.empty_qtensor(rec, 128, 256, "grad")
        state.bind(q)
        F.quantize(rec, to_dev_bf16(x), "grad", out=q)
        F.amax_update(rec, state, q.amax)
        torch.cuda.synchronize()
        ref = d.quantize(x)
        d.update(ref["amax"])
        assert np.array_equal(_np(q.row), ref["row"]), t
        assert same_f32(_np(state.scale)[0], d.scale), t
        assert same_f32(_np(state.scale_inv)[0], d.scale_inv), t


def _oracle_q(kind, b, role, delayed_scale=None):
    """The oracle's quantisation of a seeded bf16 tensor: (row deq, col deq) in float64."""
    fmt = O.hybrid_format(role)
    if kind == "tensorwise":
        q = O.quantize_tensorwise(b, fmt=fmt)
    elif kind == "delayed":
        d = O.DelayedScaling(4, fmt=fmt)
        d.scale, d.scale_inv = delayed_scale
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


@pytest.mark.parametrize("kind", ["tensorwise", "delayed", "blockwise"])
@pytest.mark.parametrize("fp32", [False, True])
# the last two shapes give dX (2560 x 4096) and dW (4096 x 2560) more tiles than the grid runs
# at once
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (2560, 256, 4096), (256, 4096, 2560)])
def test_hybrid_dgrad_wgrad(kind, fp32, M, N, K):
    """dX = dY . W and dW = dY^T . X with dY in E5M2, W and X in E4M3, against the oracle's
    GEMMs over its own quantisation of the same seeded inputs."""
    rec = F.Recipe(kind=kind, format="hybrid")
    xb = bf16_bits_normal(M, K, seed=91)
    wb = bf16_bits_normal(N, K, seed=92, sigma=0.02)
    dyb = bf16_bits_normal(M, N, seed=93, sigma=1e-3)
    qs, refs = {}, {}
    for name, b, role in (("x", xb, "activation"), ("w", wb, "weight"), ("dy", dyb, "grad")):
        q = F.empty_qtensor(rec, b.shape[0], b.shape[1], role)
        ds = None
        if kind == "delayed":                               # a scale from an earlier step
            s, si = O.scale_from_amax(O.amax_of(b) * np.float32(1.5), 0, O.hybrid_format(role))
            ds = (s, si)
            q.scale.fill_(float(s))
            q.scale_inv.fill_(float(si))
        F.quantize(rec, to_dev_bf16(b), role, out=q)
        qs[name] = q
        refs[name] = _oracle_q(kind, b, role, ds)
    dx, dw = F.linear_bwd(rec, qs["dy"], qs["x"], qs["w"], fp32=fp32)
    torch.cuda.synchronize()
    dx_ref = O.gemm_tn_f64(refs["dy"][0], refs["w"][1])
    dw_ref = O.gemm_tn_f64(refs["dy"][1], refs["x"][1])
    for got, ref in ((dx, dx_ref), (dw, dw_ref)):
        if fp32:
            ok, err = gemm_f32_normwise(_np(got), ref)
        else:
            ok, err = gemm_bf16_close(from_dev_bf16(got), ref)
        assert ok, err


@pytest.mark.parametrize("role", ["activation", "weight"])
@pytest.mark.parametrize("margin", [0, 3])
def test_blockwise_power_of_two_scales(role, margin):
    """Blockwise with power-of-two block scales: codes bit-exact, and the scales stored as E8M0
    bytes in the MXFP8 layout equal to the oracle's power-of-two s_inv."""
    rec = F.Recipe(kind="blockwise", power_2_scales=True, margin=margin)
    x = bf16_bits_normal(256, 384, seed=101, outlier_p=1e-2, outlier_factor=40.0)
    R, C = x.shape
    q = F.empty_qtensor(rec, R, C, role)
    F.quantize(rec, to_dev_bf16(x), role, out=q)
    torch.cuda.synchronize()
    if role == "weight":
        ref = O.quantize_blockwise_128x128(x, margin, pow2=True)
        rows_b = 128
    else:
        ref = O.quantize_blockwise_1x128(x, margin, pow2=True)
        rows_b = 1
    assert np.array_equal(mx_untile(_np(q.row_scale), R, C),
                          O.pow2_scales_as_e8m0(ref["row_scale_inv"], rows_b, R, C))
    assert np.array_equal(mx_untile(_np(q.col_scale), C, R),
                          O.pow2_scales_as_e8m0(ref["col_scale_inv"], rows_b, C, R))
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


@pytest.mark.parametrize("fmt", ["e4m3", "hybrid"])
@pytest.mark.parametrize("fp32", [False, True])
def test_blockwise_power_of_two_gemms(fmt, fp32):
    """fprop, dgrad and wgrad of power-of-two blockwise tensors, which run on the MXFP8
    block-scaled tensor-core path, against the oracle's blockwise GEMMs."""
    rec = F.Recipe(kind="blockwise", power_2_scales=True, format=fmt)
    M, N, K = 256, 384, 512
    xb = bf16_bits_normal(M, K, seed=102)
    wb = bf16_bits_normal(N, K, seed=103, sigma=0.02)
    dyb = bf16_bits_normal(M, N, seed=104, sigma=1e-3)
    gf = "e5m2" if fmt == "hybrid" else "e4m3"
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    wq = F.quantize(rec, to_dev_bf16(wb), "weight")
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    y = F.linear_fwd(rec, xq, wq, fp32=fp32)
    dx, dw = F.linear_bwd(rec, dyq, xq, wq, fp32=fp32)
    torch.cuda.synchronize()
    qx = O.quantize_blockwise_1x128(xb, pow2=True)
    qw = O.quantize_blockwise_128x128(wb, pow2=True)
    qd = O.quantize_blockwise_1x128(dyb, pow2=True, fmt=gf)
    refs = (
        (y, O.gemm_tn_f64(O.dequant_1x128(qx["row"], qx["row_scale_inv"]),
                          O.dequant_128x128(qw["row"], qw["row_scale_inv"]))),
        (dx, O.gemm_tn_f64(O.dequant_1x128(qd["row"], qd["row_scale_inv"], gf),
                           O.dequant_128x128(qw["col"], qw["col_scale_inv"]))),
        (dw, O.gemm_tn_f64(O.dequant_1x128(qd["col"], qd["col_scale_inv"], gf),
                           O.dequant_1x128(qx["col"], qx["col_scale_inv"]))),
    )
    for got, ref in refs:
        if fp32:
            ok, err = gemm_f32_normwise(_np(got), ref)
        else:
            ok, err = gemm_bf16_close(from_dev_bf16(got), ref)
        assert ok, err
