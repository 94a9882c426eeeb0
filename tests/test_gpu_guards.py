"""Out-of-bounds writes and tile-corner addressing, checked without a sanitizer.

1. Canaries. Every output buffer of a call (codes, scales, the per-tensor scalars, GEMM
   results, the fused MLP epilogues' copies, a grouped quantize's tensors) sits inside a
   larger allocation with 4 KiB of canary bytes on either side. After the call the canaries
   are unchanged, and the outputs equal those of the same call on plain buffers.
2. Tile corners. A tensor that is zero but for one value at a corner of a 128 x 128 tile
   (including the corners of the ragged last tile) quantises bit-exactly like the oracle,
   and its GEMM matches the oracle. An index slip at a tile edge moves or drops that value.
"""
import numpy as np
import pytest
import torch

from helpers import (bw_untile, cuda_ok, from_dev_bf16, gemm_bf16_close, mx_untile, same_f32,
                     to_dev_bf16)
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import _lib as L
    from scaled_quantize_fp8_gb300.binding import KINDS, ROLES, QTensor, scale_shape

GUARD = 4096
CANARY = 0xA5


class Guards:
    """Device buffers with canary bytes before and after each one."""

    def __init__(self):
        self.bufs = []

    def alloc(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        inner = raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            inner.fill_(fill)
        self.bufs.append((raw, n))
        return inner

    def intact(self):
        for raw, n in self.bufs:
            if bool((raw[:GUARD] != CANARY).any()) or bool((raw[GUARD + n:] != CANARY).any()):
                return False
        return True


def guarded_qtensor(g, rec, rows, cols, role, want_row=True, want_col=True):
    kind, r = KINDS[rec.kind], ROLES[role]
    q = QTensor(rows, cols, kind, r)
    if want_row:
        q.row = g.alloc((rows, cols), torch.uint8)
        shp, dt = scale_shape(kind, r, rows, cols, rec.power_2_scales)
        if shp is not None:
            q.row_scale = g.alloc(shp, dt)
    if want_col:
        if not rec.fp8_wgrad and r != L.ROLE_WEIGHT:
            q.col = g.alloc((cols, rows), torch.bfloat16)
            q.col_bf16 = 1
        else:
            q.col = g.alloc((cols, rows), torch.uint8)
            shp, dt = scale_shape(kind, r, cols, rows, rec.power_2_scales)
            if shp is not None:
                q.col_scale = g.alloc(shp, dt)
    if kind in (L.RECIPE_DELAYED, L.RECIPE_TENSORWISE):
        q.amax = g.alloc((1,), torch.float32, 0.0)
        q.scale = g.alloc((1,), torch.float32, 1.0)
        q.scale_inv = g.alloc((1,), torch.float32, 1.0)
    return q


def test_guards_see_a_stray_byte():
    """The canary check itself: one byte written just past a buffer (by torch, inside the
    guarded allocation) is reported."""
    g = Guards()
    t = g.alloc((128, 64), torch.uint8)
    assert g.intact()
    raw, n = g.bufs[0]
    raw[GUARD + n].fill_(0)
    torch.cuda.synchronize()
    assert not g.intact()
    assert t.shape == (128, 64)


FIELDS = ("row", "col", "row_scale", "col_scale", "amax", "scale", "scale_inv")


def same_qtensor(a, b):
    for f in FIELDS:
        x, y = getattr(a, f), getattr(b, f)
        if (x is None) != (y is None):
            return False
        if x is not None and not torch.equal(x.view(torch.uint8) if x.dtype != torch.uint8 else x,
                                             y.view(torch.uint8) if y.dtype != torch.uint8 else y):
            return False
    return True


QUANT_CASES = [
    ("tensorwise", "e4m3", "activation", (272, 208), {}),
    ("tensorwise", "hybrid", "grad", (144, 400), {}),
    ("tensorwise", "e4m3", "activation", (256, 384), {"fp8_wgrad": False}),
    ("delayed", "e4m3", "activation", (528, 48), {}),
    ("mxfp8", "e4m3", "activation", (256, 384), {}),
    ("mxfp8", "e4m3", "weight", (384, 128), {}),
    ("blockwise", "e4m3", "activation", (256, 384), {}),
    ("blockwise", "e4m3", "weight", (384, 256), {}),
    ("blockwise", "hybrid", "grad", (128, 512), {"power_2_scales": True}),
]


@pytest.mark.parametrize("kind,fmt,role,shape,extra", QUANT_CASES)
def test_quantize_writes_stay_inside(kind, fmt, role, shape, extra):
    rec = F.Recipe(kind=kind, format=fmt, **extra)
    R, C = shape
    x = to_dev_bf16(bf16_bits_normal(R, C, seed=130, outlier_p=1e-2, outlier_factor=30.0))
    g = Guards()
    q = guarded_qtensor(g, rec, R, C, role)
    ref = F.empty_qtensor(rec, R, C, role)
    F.quantize(rec, x, role, out=q)
    F.quantize(rec, x, role, out=ref)
    torch.cuda.synchronize()
    assert g.intact()
    assert same_qtensor(q, ref)


@pytest.mark.parametrize("kind,extra", [("mxfp8", {}), ("blockwise", {}),
                                         ("blockwise", {"format": "hybrid", "power_2_scales": True})])
@pytest.mark.parametrize("fp8_wgrad", [True, False])
def test_quantize_group_writes_stay_inside(kind, extra, fp8_wgrad):
    # one grouped launch over three tensors of different tile counts (blockwise: 1x128, 128x128
    # and a 1x128 gradient, E5M2 under the hybrid format)
    rec = F.Recipe(kind=kind, fp8_wgrad=fp8_wgrad, **extra)
    shapes, roles = [(256, 384), (384, 128), (128, 512)], ["activation", "weight", "grad"]
    xs = [to_dev_bf16(bf16_bits_normal(r, c, seed=140 + i, outlier_p=1e-2, outlier_factor=30.0))
          for i, (r, c) in enumerate(shapes)]
    g = Guards()
    qs = [guarded_qtensor(g, rec, r, c, role) for (r, c), role in zip(shapes, roles)]
    F.quantize_group(rec, xs, roles, outs=qs)
    refs = [F.quantize(rec, x, role) for x, role in zip(xs, roles)]
    torch.cuda.synchronize()
    assert g.intact()
    for q, ref in zip(qs, refs):
        assert same_qtensor(q, ref)


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
@pytest.mark.parametrize("fp32", [False, True])
def test_gemm_writes_stay_inside(kind, fp32):
    rec = F.Recipe(kind=kind)
    M, N, K = 384, 384, 256               # a full and a partial tile in M and in N
    xq = F.quantize(rec, to_dev_bf16(bf16_bits_normal(M, K, seed=131)), "activation")
    wq = F.quantize(rec, to_dev_bf16(bf16_bits_normal(N, K, seed=132, sigma=0.02)), "weight")
    dyq = F.quantize(rec, to_dev_bf16(bf16_bits_normal(M, N, seed=133, sigma=1e-3)), "grad")
    dt = torch.float32 if fp32 else torch.bfloat16
    g = Guards()
    y, dx, dw = g.alloc((M, N), dt), g.alloc((M, K), dt), g.alloc((N, K), dt)
    F.linear_fwd(rec, xq, wq, y=y, fp32=fp32)
    F.linear_bwd(rec, dyq, xq, wq, dx=dx, dw=dw, fp32=fp32)
    y_ref = F.linear_fwd(rec, xq, wq, fp32=fp32)
    dx_ref, dw_ref = F.linear_bwd(rec, dyq, xq, wq, fp32=fp32)
    torch.cuda.synchronize()
    assert g.intact()
    for a, b in ((y, y_ref), (dx, dx_ref), (dw, dw_ref)):
        assert torch.equal(a, b)


def test_fused_mlp_writes_stay_inside():
    rec = F.Recipe(kind="mxfp8")
    M, H, Fd = 384, 256, 640
    xq = F.quantize(rec, to_dev_bf16(bf16_bits_normal(M, H, seed=134)), "activation")
    w1q = F.quantize(rec, to_dev_bf16(bf16_bits_normal(Fd, H, seed=135, sigma=0.02)), "weight")
    w2q = F.quantize(rec, to_dev_bf16(bf16_bits_normal(H, Fd, seed=136, sigma=0.02)), "weight")
    dyq = F.quantize(rec, to_dev_bf16(bf16_bits_normal(M, H, seed=137, sigma=1e-3)), "grad")
    g = Guards()
    a_q = guarded_qtensor(g, rec, M, Fd, "activation")
    h_q = guarded_qtensor(g, rec, M, Fd, "activation", want_col=False)
    dh_q = guarded_qtensor(g, rec, M, Fd, "grad")
    F.linear_fwd_gelu(rec, xq, w1q, a_q=a_q, h_q=h_q)
    F.linear_dgrad_dgelu(rec, dyq, w2q, h_q, dh_q=dh_q)
    a_ref, h_ref = F.linear_fwd_gelu(rec, xq, w1q)
    dh_ref = F.linear_dgrad_dgelu(rec, dyq, w2q, h_ref)
    torch.cuda.synchronize()
    assert g.intact()
    assert same_qtensor(a_q, a_ref) and same_qtensor(h_q, h_ref) and same_qtensor(dh_q, dh_ref)


def _corners(R, C):
    """Corners of the first tile, of an inner tile and of the last (possibly ragged) tile."""
    pts = {(0, 0), (0, 127), (127, 0), (127, 127), (R - 1, C - 1), (R - 1, 0), (0, C - 1)}
    if R > 128 and C > 128:
        pts |= {(128, 128), (min(R, 256) - 1, min(C, 256) - 1)}
    return sorted(pts)


def _one_hot(R, C, r, c, value_bits=0x4170):        # bf16 15.0
    x = np.zeros((R, C), dtype=np.uint16)
    x[r, c] = value_bits
    return x


@pytest.mark.parametrize("kind,role,shape", [("tensorwise", "activation", (272, 208)),
                                             ("mxfp8", "activation", (256, 384)),
                                             ("blockwise", "activation", (256, 384)),
                                             ("blockwise", "weight", (384, 256))])
def test_single_value_at_tile_corners_quantizes_exactly(kind, role, shape):
    R, C = shape
    rec = F.Recipe(kind=kind)
    for r, c in _corners(R, C):
        x = _one_hot(R, C, r, c)
        q = F.quantize(rec, to_dev_bf16(x), role)
        torch.cuda.synchronize()
        row, col = q.row.cpu().numpy(), q.col.cpu().numpy()
        if kind == "tensorwise":
            ref = O.quantize_tensorwise(x)
            assert same_f32(q.scale_inv.cpu().numpy()[0], ref["scale_inv"]), (r, c)
        elif kind == "mxfp8":
            ref = O.quantize_mxfp8(x)
            assert np.array_equal(mx_untile(q.row_scale.cpu().numpy(), R, C), ref["row_scale"])
            assert np.array_equal(mx_untile(q.col_scale.cpu().numpy(), C, R), ref["col_scale"])
        elif role == "weight":
            ref = O.quantize_blockwise_128x128(x)
            assert np.array_equal(q.row_scale.cpu().numpy(), ref["row_scale_inv"]), (r, c)
        else:
            ref = O.quantize_blockwise_1x128(x)
            assert np.array_equal(bw_untile(q.row_scale.cpu().numpy(), R, C),
                                  ref["row_scale_inv"]), (r, c)
            assert np.array_equal(bw_untile(q.col_scale.cpu().numpy(), C, R),
                                  ref["col_scale_inv"]), (r, c)
        assert np.array_equal(row, ref["row"]), (r, c)
        assert np.array_equal(col, ref["col"]), (r, c)
        assert np.count_nonzero(row) == 1 and row[r, c] != 0, (r, c)


@pytest.mark.parametrize("kind", ["tensorwise", "mxfp8", "blockwise"])
def test_single_value_at_tile_corners_multiplies_exactly(kind):
    """X zero but for one value: Y = X W^T is that value times one row of W, placed in the row
    of the value. Each corner of X's tiles (its K dimension is W's K) goes through the GEMM."""
    M, N, K = 256, 384, 384
    rec = F.Recipe(kind=kind)
    wb = bf16_bits_normal(N, K, seed=138, sigma=0.02)
    wq = F.quantize(rec, to_dev_bf16(wb), "weight")
    if kind == "mxfp8":
        qw = O.quantize_mxfp8(wb, want_col=False)
        w_deq = O.dequant_mx(qw["row"], qw["row_scale"])
    elif kind == "tensorwise":
        qw = O.quantize_tensorwise(wb)
        w_deq = O.dequant_tensor(qw["row"], qw["scale_inv"])
    else:
        qw = O.quantize_blockwise_128x128(wb)
        w_deq = O.dequant_128x128(qw["row"], qw["row_scale_inv"])
    for r, c in _corners(M, K):
        x = _one_hot(M, K, r, c)
        xq = F.quantize(rec, to_dev_bf16(x), "activation")
        y = F.linear_fwd(rec, xq, wq)
        torch.cuda.synchronize()
        if kind == "mxfp8":
            qx = O.quantize_mxfp8(x, want_col=False)
            x_deq = O.dequant_mx(qx["row"], qx["row_scale"])
        elif kind == "tensorwise":
            qx = O.quantize_tensorwise(x)
            x_deq = O.dequant_tensor(qx["row"], qx["scale_inv"])
        else:
            qx = O.quantize_blockwise_1x128(x)
            x_deq = O.dequant_1x128(qx["row"], qx["row_scale_inv"])
        ref = O.gemm_tn_f64(x_deq, w_deq)
        got = from_dev_bf16(y)
        ok, err = gemm_bf16_close(got, ref)
        assert ok, (r, c, err)
        others = np.delete(got, r, axis=0)
        assert not np.any(others & 0x7FFF), (r, c)          # every other row is exactly zero
