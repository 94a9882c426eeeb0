"""GPU parity of the scaled FP8 GEMMs (fprop, dgrad, wgrad) against the oracle's fp64 sums.

The oracle quantises the same seeded bf16 inputs itself (its codes are independently pinned and
the GPU's are checked bit-exact in test_gpu_quantize), dequantises, and sums in float64. GPU
bf16 outputs must agree elementwise within 1e-2 relative error (floor 1e-3 of the output's
max); the fp32-output mode must agree normwise within 1e-5.
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close, gemm_f32_normwise, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _quant_gpu(rec, bits, role):
    x = to_dev_bf16(bits)
    q = F.quantize(rec, x, role)
    return q


def _oracle_deq(kind, bits, role, copy):
    """Dequantised row ('row') or column ('col') copy by the oracle, float64."""
    if kind == "tensorwise":
        q = O.quantize_tensorwise(bits)
        return O.dequant_tensor(q[copy], q["scale_inv"])
    if kind == "mxfp8":
        q = O.quantize_mxfp8(bits)
        return O.dequant_mx(q[copy], q[copy + "_scale"])
    if role == "weight":
        q = O.quantize_blockwise_128x128(bits)
        return O.dequant_128x128(q[copy], q[copy + "_scale_inv"])
    q = O.quantize_blockwise_1x128(bits)
    return O.dequant_1x128(q[copy], q[copy + "_scale_inv"])


def _check(got, ref, fp32):
    if fp32:
        ok, err = gemm_f32_normwise(got.cpu().numpy(), ref)
    else:
        ok, err = gemm_bf16_close(from_dev_bf16(got), ref)
    assert ok, f"error {err}"
    return err


SHAPES_SMALL = [(256, 256, 256), (384, 512, 512), (128, 768, 384), (640, 256, 1024)]


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
@pytest.mark.parametrize("M,N,K", SHAPES_SMALL)
@pytest.mark.parametrize("fp32", [False, True])
def test_fprop(kind, M, N, K, fp32):
    rec = F.Recipe(kind=kind)
    xb = bf16_bits_normal(M, K, seed=11, outlier_p=1e-3 if kind == "mxfp8" else 0.0)
    wb = bf16_bits_normal(N, K, seed=12, sigma=0.02)
    xq = _quant_gpu(rec, xb, "activation")
    wq = _quant_gpu(rec, wb, "weight")
    y = F.linear_fwd(rec, xq, wq, fp32=fp32)
    torch.cuda.synchronize()
    ref = O.gemm_tn_f64(_oracle_deq(kind, xb, "activation", "row"),
                        _oracle_deq(kind, wb, "weight", "row"))
    _check(y, ref, fp32)


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
# the last two shapes give dgrad (dX 2560 x 4096) and wgrad (dW 4096 x 2560) more tiles than
# the grid runs at once
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (512, 256, 128), (2560, 256, 4096),
                                   (256, 4096, 2560)])
@pytest.mark.parametrize("fp32", [False, True])
def test_dgrad_wgrad(kind, M, N, K, fp32):
    rec = F.Recipe(kind=kind)
    xb = bf16_bits_normal(M, K, seed=13)
    wb = bf16_bits_normal(N, K, seed=14, sigma=0.02)
    dyb = bf16_bits_normal(M, N, seed=15, sigma=1e-3)
    xq = _quant_gpu(rec, xb, "activation")
    wq = _quant_gpu(rec, wb, "weight")
    dyq = _quant_gpu(rec, dyb, "grad")
    dx, dw = F.linear_bwd(rec, dyq, xq, wq, fp32=fp32)
    torch.cuda.synchronize()
    ref_dx = O.gemm_tn_f64(_oracle_deq(kind, dyb, "grad", "row"),
                           _oracle_deq(kind, wb, "weight", "col"))
    ref_dw = O.gemm_tn_f64(_oracle_deq(kind, dyb, "grad", "col"),
                           _oracle_deq(kind, xb, "activation", "col"))
    _check(dx, ref_dx, fp32)
    _check(dw, ref_dw, fp32)


# More tiles than the persistent grid runs at once: 160 pair tiles on 76 pairs (tensorwise,
# MXFP8) or 320 single-CTA tiles on 152 SMs (blockwise), so the last round is partial; with
# M > N the tile groups run along N (the exchanged order), with M < N along M. Every element
# is compared, in bf16 and in fp32 output mode.
@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
@pytest.mark.parametrize("M,N", [(4096, 2560), (2560, 4096)])
def test_fprop_multi_round_full_compare(kind, M, N):
    K = 256
    rec = F.Recipe(kind=kind)
    xb = bf16_bits_normal(M, K, seed=17, outlier_p=1e-3 if kind == "mxfp8" else 0.0)
    wb = bf16_bits_normal(N, K, seed=18, sigma=0.02)
    xq = _quant_gpu(rec, xb, "activation")
    wq = _quant_gpu(rec, wb, "weight")
    y = F.linear_fwd(rec, xq, wq)
    y32 = F.linear_fwd(rec, xq, wq, fp32=True)
    torch.cuda.synchronize()
    ref = O.gemm_tn_f64(_oracle_deq(kind, xb, "activation", "row"),
                        _oracle_deq(kind, wb, "weight", "row"))
    _check(y, ref, False)
    _check(y32, ref, True)


@pytest.mark.parametrize("M,N,K", [(272, 208, 144), (16, 16, 16), (400, 528, 48)])
def test_tensorwise_ragged(M, N, K):
    rec = F.Recipe(kind="tensorwise")
    xb = bf16_bits_normal(M, K, seed=16)
    wb = bf16_bits_normal(N, K, seed=17)
    y = F.linear_fwd(rec, _quant_gpu(rec, xb, "activation"), _quant_gpu(rec, wb, "weight"))
    y32 = F.linear_fwd(rec, _quant_gpu(rec, xb, "activation"), _quant_gpu(rec, wb, "weight"),
                       fp32=True)
    torch.cuda.synchronize()
    ref = O.gemm_tn_f64(_oracle_deq("tensorwise", xb, "activation", "row"),
                        _oracle_deq("tensorwise", wb, "weight", "row"))
    _check(y, ref, False)
    _check(y32, ref, True)


def test_config1_tensorwise_256():
    """Tensorwise quantize of X, W 256 x 256 N(0,1), seed 0, margin 0, then Y = X W^T."""
    rec = F.Recipe(kind="tensorwise")
    xb = bf16_bits_normal(256, 256, seed=0, stream=0)
    wb = bf16_bits_normal(256, 256, seed=0, stream=1)
    xq, wq = _quant_gpu(rec, xb, "activation"), _quant_gpu(rec, wb, "weight")
    y = F.linear_fwd(rec, xq, wq)
    y32 = F.linear_fwd(rec, xq, wq, fp32=True)
    torch.cuda.synchronize()
    ref = O.gemm_tn_f64(_oracle_deq("tensorwise", xb, "activation", "row"),
                        _oracle_deq("tensorwise", wb, "weight", "row"))
    _check(y, ref, False)
    _check(y32, ref, True)


def test_zero_k_gives_zeros():
    rec = F.Recipe(kind="tensorwise")
    xq = F.quantize(rec, torch.zeros((128, 0), dtype=torch.bfloat16, device="cuda"),
                    out=F.empty_qtensor(rec, 128, 0))
    wq = F.quantize(rec, torch.zeros((64, 0), dtype=torch.bfloat16, device="cuda"),
                    out=F.empty_qtensor(rec, 64, 0))
    xq.row = torch.empty((128, 16), dtype=torch.uint8, device="cuda")   # any valid pointer
    wq.row = torch.empty((64, 16), dtype=torch.uint8, device="cuda")
    y = torch.full((128, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    F.linear_fwd(rec, xq, wq, y=y)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def _sample_rows(M, n=256):
    g = np.random.default_rng(5)
    rows = np.concatenate([np.arange(128), np.arange(M - 128, M), g.choice(M, n, replace=False)])
    return np.unique(rows)


def test_full_size_mxfp8_fprop_sampled():
    """MXFP8 fprop 8192 x 4096 x 4096 in the benchmark's launch configuration; the oracle sums
    a sample of output rows (first and last tiles plus random rows)."""
    rec = F.Recipe(kind="mxfp8")
    xb = bf16_bits_normal(8192, 4096, seed=0, stream=0, outlier_p=1e-3, outlier_factor=50.0)
    wb = bf16_bits_normal(4096, 4096, seed=0, stream=1, sigma=0.02)
    xq, wq = _quant_gpu(rec, xb, "activation"), _quant_gpu(rec, wb, "weight")
    y = F.linear_fwd(rec, xq, wq)
    y32 = F.linear_fwd(rec, xq, wq, fp32=True)
    torch.cuda.synchronize()
    rows = _sample_rows(8192)
    qx, qw = O.quantize_mxfp8(xb[rows], want_col=False), O.quantize_mxfp8(wb, want_col=False)
    ref = O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                        O.dequant_mx(qw["row"], qw["row_scale"]))
    ok, err = gemm_bf16_close(from_dev_bf16(y)[rows], ref)
    assert ok, err
    ok, err = gemm_f32_normwise(y32.cpu().numpy()[rows], ref)
    assert ok, err


# ------------------------------------------------------------------ --fp8-wgrad off

@pytest.mark.parametrize("kind", ["tensorwise", "delayed", "mxfp8", "blockwise"])
# the last shape's dW (4096 x 2560) has more tiles than the grid runs at once
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (512, 256, 128), (640, 512, 384), (256, 128, 256),
                                   (256, 4096, 2560)])
@pytest.mark.parametrize("fp32", [False, True])
def test_wgrad_bf16(kind, M, N, K, fp32):
    """With fp8_wgrad off the column copies of X and dY are bf16 transposes and wgrad is a
    bf16 GEMM: dW = dY^T X summed in fp32, against the oracle's fp64 sum of the bf16 values."""
    rec = F.Recipe(kind=kind, fp8_wgrad=False)
    xb = bf16_bits_normal(M, K, seed=51)
    dyb = bf16_bits_normal(M, N, seed=52, sigma=1e-3)
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    assert xq.col_bf16 == 1 and np.array_equal(from_dev_bf16(xq.col), xb.T)
    assert np.array_equal(from_dev_bf16(dyq.col), dyb.T)
    _, dw = F.linear_bwd(rec, dyq, xq, None, want_dx=False, fp32=fp32)
    torch.cuda.synchronize()
    ref = O.bf16_gemm_tn_f64(np.ascontiguousarray(dyb.T), np.ascontiguousarray(xb.T))
    _check(dw, ref, fp32)


def test_wgrad_bf16_with_fp8_dgrad():
    """Mixed backward: dgrad stays FP8 (weight column copy) while wgrad runs in bf16."""
    rec = F.Recipe(kind="mxfp8", fp8_wgrad=False)
    M, N, K = 384, 256, 512
    xb = bf16_bits_normal(M, K, seed=53)
    wb = bf16_bits_normal(N, K, seed=54, sigma=0.02)
    dyb = bf16_bits_normal(M, N, seed=55, sigma=1e-3)
    xq, wq, dyq = (F.quantize(rec, to_dev_bf16(b), r)
                   for b, r in ((xb, "activation"), (wb, "weight"), (dyb, "grad")))
    assert wq.col_bf16 == 0
    dx, dw = F.linear_bwd(rec, dyq, xq, wq)
    torch.cuda.synchronize()
    _check(dx, O.gemm_tn_f64(_oracle_deq("mxfp8", dyb, "grad", "row"),
                             _oracle_deq("mxfp8", wb, "weight", "col")), False)
    _check(dw, O.bf16_gemm_tn_f64(np.ascontiguousarray(dyb.T), np.ascontiguousarray(xb.T)), False)


def test_full_size_blockwise_fwd_dgrad_wgrad_sampled():
    """Blockwise fwd + dgrad + wgrad at 4096 x 4096 x 4096 (X 1x128, W 128x128, dY N(0,1e-3)),
    in the benchmark's launch configuration, in bf16 and fp32 output mode; the oracle sums
    sampled output rows."""
    rec = F.Recipe(kind="blockwise")
    xb = bf16_bits_normal(4096, 4096, seed=0, stream=0)
    wb = bf16_bits_normal(4096, 4096, seed=0, stream=1, sigma=0.02)
    dyb = bf16_bits_normal(4096, 4096, seed=0, stream=2, sigma=1e-3)
    xq, wq, dyq = (F.quantize(rec, to_dev_bf16(b), r)
                   for b, r in ((xb, "activation"), (wb, "weight"), (dyb, "grad")))
    y = F.linear_fwd(rec, xq, wq)
    dx, dw = F.linear_bwd(rec, dyq, xq, wq)
    y32 = F.linear_fwd(rec, xq, wq, fp32=True)
    dx32, dw32 = F.linear_bwd(rec, dyq, xq, wq, fp32=True)
    torch.cuda.synchronize()
    rows = _sample_rows(4096)
    qx, qw, qd = (O.quantize_blockwise_1x128(xb), O.quantize_blockwise_128x128(wb),
                  O.quantize_blockwise_1x128(dyb))
    d1 = lambda q, c: O.dequant_1x128(q[c], q[c + "_scale_inv"])  # noqa: E731
    d2 = lambda q, c: O.dequant_128x128(q[c], q[c + "_scale_inv"])  # noqa: E731
    for got, got32, a, b in ((y, y32, d1(qx, "row"), d2(qw, "row")),
                             (dx, dx32, d1(qd, "row"), d2(qw, "col")),
                             (dw, dw32, d1(qd, "col"), d1(qx, "col"))):
        ref = O.gemm_tn_f64(a[rows], b)
        ok, err = gemm_bf16_close(from_dev_bf16(got)[rows], ref)
        assert ok, err
        # the promoted fp32 sum (per 128-wide K chunk, times both block scales) agrees with
        # the fp64 sum on the same FP8 operands
        ok, err = gemm_f32_normwise(got32.cpu().numpy()[rows], ref)
        assert ok, ("fp32", err)
