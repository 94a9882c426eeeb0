"""GPU parity of the fp32 master-weight quantizer (fp8_quantize_master): every recipe's codes
and scales bit-exact against the oracle fed the same fp32 values, including values bf16 cannot
hold (no bf16 rounding on the way), ragged per-tensor shapes, special values, and agreement with
the bf16 quantizer on fp32 inputs that bf16 holds exactly."""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, mx_untile, same_f32, to_dev_bf16
from oracle import fp8_oracle as O

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _np(t):
    return t.cpu().numpy()


def _w32(R, C, seed, sigma=0.02):
    return (np.random.default_rng(seed).standard_normal((R, C)) * sigma).astype(np.float32)


def _check(kind, w, margin=0, delayed_scale=None):
    R, C = w.shape
    rec = F.Recipe(kind=kind, margin=margin)
    out = F.empty_qtensor(rec, R, C, "weight")
    if delayed_scale is not None:
        out.scale.fill_(float(delayed_scale))
        out.scale_inv.fill_(float(np.float32(1.0) / np.float32(delayed_scale)))
    F.quantize_master(rec, torch.from_numpy(w).cuda(), out=out)
    torch.cuda.synchronize()
    if kind == "tensorwise":
        ref = O.quantize_tensorwise(w, margin)
        assert same_f32(_np(out.amax)[0], ref["amax"])
        assert same_f32(_np(out.scale)[0], ref["scale"])
        assert same_f32(_np(out.scale_inv)[0], ref["scale_inv"])
    elif kind == "delayed":
        d = O.DelayedScaling(4, margin)
        d.scale = np.float32(delayed_scale)
        ref = d.quantize(w)
        assert same_f32(_np(out.amax)[0], ref["amax"])
    elif kind == "mxfp8":
        ref = O.quantize_mxfp8(w)
        assert np.array_equal(mx_untile(_np(out.row_scale), R, C), ref["row_scale"])
        assert np.array_equal(mx_untile(_np(out.col_scale), C, R), ref["col_scale"])
    else:
        ref = O.quantize_blockwise_128x128(w, margin)
        assert np.array_equal(_np(out.row_scale), ref["row_scale_inv"])
        assert np.array_equal(_np(out.col_scale), ref["col_scale_inv"])
    assert np.array_equal(_np(out.row), ref["row"])
    assert np.array_equal(_np(out.col), ref["col"])
    return out


@pytest.mark.parametrize("kind", ["tensorwise", "delayed", "mxfp8", "blockwise"])
@pytest.mark.parametrize("shape", [(256, 384), (384, 128)])
def test_master_tiles(kind, shape):
    w = _w32(*shape, seed=shape[0] + shape[1])
    _check(kind, w, delayed_scale=np.float32(1000.0) if kind == "delayed" else None)


@pytest.mark.parametrize("kind", ["tensorwise", "delayed"])
@pytest.mark.parametrize("shape", [(144, 208), (16, 16), (272, 48)])
def test_master_ragged_per_tensor(kind, shape):
    _check(kind, _w32(*shape, seed=7), margin=1,
           delayed_scale=np.float32(3000.0) if kind == "delayed" else None)


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
def test_master_special_values(kind):
    w = _w32(256, 256, seed=9, sigma=1.0)
    w[0, :32] = 0.0
    w[1, 3] = np.float32(1e-41)                  # fp32 subnormal
    w[2, 7] = np.float32(3e38)
    w[130, 5] = np.inf
    w[200, 201] = -np.inf
    w[250, 100] = np.nan
    w[40, 41] = -0.0
    _check(kind, w)


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
def test_master_matches_bf16_path_on_bf16_values(kind):
    """fp32 inputs that bf16 holds exactly give the bf16 quantizer's bytes."""
    wb = O.f64_to_bf16(_w32(256, 384, seed=11).astype(np.float64))
    w = O.bf16_to_f32(wb)
    rec = F.Recipe(kind=kind)
    qm = F.quantize_master(rec, torch.from_numpy(w).cuda())
    qb = F.quantize(rec, to_dev_bf16(wb), "weight")
    torch.cuda.synchronize()
    for f in ("row", "col", "row_scale", "col_scale", "scale", "scale_inv"):
        a, b = getattr(qm, f), getattr(qb, f)
        if a is not None:
            assert torch.equal(a, b), f


def test_master_full_size_mxfp8_weight():
    """W 4096 x 4096 fp32 master weight, MXFP8 row and column copies."""
    _check("mxfp8", _w32(4096, 4096, seed=13))
