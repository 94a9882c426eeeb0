"""GPU parity of the quantize-cast kernels against the oracle: bit-exact codes and scales.

Covers every recipe on multi-tile shapes, ragged tails (per-tensor recipes accept multiples of
16), the exhaustive sweep of all 65,536 bf16 bit patterns at several scales, edge tensors
(zeros, one outlier, signed zeros, subnormals, saturation, NaN/Inf), an empty tensor, and the
full-size workload shapes (X 8192 x 4096, W 4096 x 4096) in the launch configuration the
benchmark uses.
"""
import numpy as np
import pytest
import torch

from helpers import bw_untile, cuda_ok, mx_untile, same_f32, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_from_f32, bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _q(kind, x_bits, role="activation", margin=0, want_row=True, want_col=True, scale=None):
    rec = F.Recipe(kind=kind, margin=margin)
    x = to_dev_bf16(x_bits)
    out = F.empty_qtensor(rec, x.shape[0], x.shape[1], role, want_row, want_col)
    if scale is not None:                     # delayed: the scale the history produced
        out.scale.fill_(float(scale))
        out.scale_inv.fill_(float(np.float32(1.0) / np.float32(scale)))
    F.quantize(rec, x, role, want_row, want_col, out=out)
    torch.cuda.synchronize()
    return out


def _np(t):
    return t.cpu().numpy()


def check_tensorwise(x_bits, margin=0):
    q = _q("tensorwise", x_bits, margin=margin)
    ref = O.quantize_tensorwise(x_bits, margin)
    assert same_f32(_np(q.amax)[0], ref["amax"])
    assert same_f32(_np(q.scale)[0], ref["scale"])
    assert same_f32(_np(q.scale_inv)[0], ref["scale_inv"])
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


def check_delayed(x_bits, scale):
    q = _q("delayed", x_bits, scale=scale)
    d = O.DelayedScaling(4)
    d.scale = np.float32(scale)
    ref = d.quantize(x_bits)
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])
    assert same_f32(_np(q.amax)[0], ref["amax"])


def check_mx(x_bits):
    R, C = x_bits.shape
    q = _q("mxfp8", x_bits)
    ref = O.quantize_mxfp8(x_bits)
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(mx_untile(_np(q.row_scale), R, C), ref["row_scale"])
    assert np.array_equal(_np(q.col), ref["col"])
    assert np.array_equal(mx_untile(_np(q.col_scale), C, R), ref["col_scale"])


def check_bw(x_bits, role, margin=0):
    R, C = x_bits.shape
    q = _q("blockwise", x_bits, role=role, margin=margin)
    if role == "weight":
        ref = O.quantize_blockwise_128x128(x_bits, margin)
        assert np.array_equal(_np(q.row_scale), ref["row_scale_inv"])
        assert np.array_equal(_np(q.col_scale), ref["col_scale_inv"])
    else:
        ref = O.quantize_blockwise_1x128(x_bits, margin)
        assert np.array_equal(bw_untile(_np(q.row_scale), R, C), ref["row_scale_inv"])
        assert np.array_equal(bw_untile(_np(q.col_scale), C, R), ref["col_scale_inv"])
    assert np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(_np(q.col), ref["col"])


# ------------------------------------------------------------------ multi-tile shapes

@pytest.mark.parametrize("shape", [(256, 384), (384, 128), (128, 640)])
def test_tensorwise_tiles(shape):
    check_tensorwise(bf16_bits_normal(*shape, seed=1))
    check_tensorwise(bf16_bits_normal(*shape, seed=2, sigma=1e-3), margin=3)


@pytest.mark.parametrize("shape", [(272, 208), (16, 16), (144, 400), (528, 48)])
def test_tensorwise_ragged(shape):
    check_tensorwise(bf16_bits_normal(*shape, seed=3, sigma=4.0))


@pytest.mark.parametrize("shape", [(256, 384), (272, 208)])
@pytest.mark.parametrize("scale", [1.0, 448.0 / 3.0, 2.0 ** -7, 1e20])
def test_delayed_cast(shape, scale):
    check_delayed(bf16_bits_normal(*shape, seed=4), scale)


@pytest.mark.parametrize("shape", [(256, 384), (128, 128), (384, 256)])
def test_mxfp8_tiles(shape):
    check_mx(bf16_bits_normal(*shape, seed=5, outlier_p=1e-2))


@pytest.mark.parametrize("shape", [(256, 384), (128, 128), (384, 256)])
@pytest.mark.parametrize("role", ["activation", "weight", "grad"])
def test_blockwise_tiles(shape, role):
    check_bw(bf16_bits_normal(*shape, seed=6, sigma=0.02), role)
    check_bw(bf16_bits_normal(*shape, seed=7), role, margin=2)


# ------------------------------------------------------------------ exhaustive bf16 sweep

def _all_bf16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)


@pytest.mark.parametrize("scale", [1.0, 448.0, 2.0 ** -7, 1.0 / 3.0, 3.0, 1e-30, 1e30])
def test_exhaustive_bf16_cast(scale):
    check_delayed(_all_bf16(), scale)


def test_exhaustive_bf16_all_recipes():
    x = _all_bf16()
    check_tensorwise(x)                       # contains NaN -> amax NaN -> scale 1
    check_mx(x)
    check_bw(x, "activation")
    check_bw(x, "weight")
    # a permuted sweep mixes magnitudes inside every block
    perm = np.random.default_rng(0).permutation(65536)
    xp = _all_bf16().reshape(-1)[perm].reshape(256, 256)
    check_mx(xp)
    check_bw(xp, "activation")


# ------------------------------------------------------------------ edge tensors

def _edge_cases():
    z = np.zeros((128, 256), np.float32)
    one = z.copy()
    one[77, 201] = 12345.0
    signed0 = z.copy()
    signed0[::2, ::3] = -0.0
    sub = np.full((128, 256), 1e-39, np.float32) * np.sign(np.random.default_rng(1).standard_normal((128, 256)))
    sat = np.random.default_rng(2).uniform(440, 480, (128, 256)).astype(np.float32)
    ties = np.tile(np.array([1.0625, 1.1875, 248.0, 232.0, -1.0625, 2.0 ** -10], np.float32),
                   (128, 43))[:, :256]
    inf = np.random.default_rng(3).standard_normal((128, 256)).astype(np.float32)
    inf[5, 5] = np.inf
    inf[100, 200] = -np.inf
    nan = np.random.default_rng(4).standard_normal((128, 256)).astype(np.float32)
    nan[64, 31] = np.nan
    return {"zeros": z, "outlier": one, "signed_zero": signed0, "subnormal": sub,
            "saturation": sat, "ties": ties, "inf": inf, "nan": nan}


@pytest.mark.parametrize("case", list(_edge_cases().keys()))
def test_edge_tensors(case):
    x = bf16_bits_from_f32(_edge_cases()[case])
    check_tensorwise(x)
    check_tensorwise(x, margin=5)
    check_delayed(x, 448.0)
    check_mx(x)
    check_bw(x, "activation")
    check_bw(x, "weight")


def test_empty_tensor_tensorwise():
    rec = F.Recipe(kind="tensorwise")
    q = F.empty_qtensor(rec, 0, 128)
    q.amax.fill_(7.0)
    q.scale.fill_(7.0)
    F.quantize(rec, torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"), out=q)
    torch.cuda.synchronize()
    assert q.amax.item() == 0.0 and q.scale.item() == 1.0 and q.scale_inv.item() == 1.0


def test_only_one_copy():
    x = bf16_bits_normal(256, 384, seed=8)
    ref = O.quantize_mxfp8(x)
    q = _q("mxfp8", x, want_col=False)
    assert q.col is None and np.array_equal(_np(q.row), ref["row"])
    assert np.array_equal(mx_untile(_np(q.row_scale), 256, 384), ref["row_scale"])
    q = _q("mxfp8", x, want_row=False)
    assert np.array_equal(_np(q.col), ref["col"])


# ------------------------------------------------------------------ full-size workloads

def test_full_size_mxfp8_x_and_w():
    x = bf16_bits_normal(8192, 4096, seed=0, outlier_p=1e-3, outlier_factor=50.0)
    check_mx(x)
    w = bf16_bits_normal(4096, 4096, seed=0, stream=1, sigma=0.02)
    check_mx(w)


def test_full_size_blockwise_and_tensorwise():
    x = bf16_bits_normal(4096, 4096, seed=0)
    check_bw(x, "activation")
    w = bf16_bits_normal(4096, 4096, seed=0, stream=1, sigma=0.02)
    check_bw(w, "weight")
    check_tensorwise(x)


def test_full_size_delayed_x():
    x = bf16_bits_normal(8192, 4096, seed=0, stream=100, sigma=2.5)
    check_delayed(x, 448.0 / 9.0)
