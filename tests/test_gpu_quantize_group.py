"""GPU parity of fp8_quantize_group (several MXFP8 or blockwise tensors in one launch).

The grouped call must write exactly the bytes that fp8_quantize writes for each tensor on its
own: codes and E8M0 scales of both copies, or the bf16 column transpose with --fp8-wgrad off.
Checked on groups of mixed shapes and roles (different tile counts, so one CTA's walk crosses
from one tensor into the next), on an empty member, on four members, on the MLP step's own
X 8192 x 4096, W1 16384 x 4096 and W2 4096 x 16384 at full size, and on a small group against
the oracle directly; blockwise groups mix 1x128 and 128x128 members, under the hybrid format,
power-of-two scales, --fp8-wgrad off and a margin.
"""
import numpy as np
import pytest
import torch

from helpers import bw_untile, cuda_ok, mx_untile, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F

FIELDS = ("row", "row_scale", "col", "col_scale")


def _bytes(t):
    return None if t is None else t.view(torch.uint8).cpu().numpy()


def _group_vs_single(shapes, roles, fp8_wgrad=True, sigmas=None, streams=None):
    rec = F.Recipe(kind="mxfp8", fp8_wgrad=fp8_wgrad)
    sigmas = sigmas or [1.0] * len(shapes)
    streams = streams or list(range(10, 10 + len(shapes)))
    xs = [to_dev_bf16(bf16_bits_normal(r, c, sigma=s, seed=3, stream=st))
          for (r, c), s, st in zip(shapes, sigmas, streams)]
    got = F.quantize_group(rec, xs, roles)
    want = [F.quantize(rec, x, r) for x, r in zip(xs, roles)]
    torch.cuda.synchronize()
    for i, (g, w) in enumerate(zip(got, want)):
        assert (g.rows, g.cols, g.kind, g.role, g.col_bf16) == \
            (w.rows, w.cols, w.kind, w.role, w.col_bf16), i
        for f in FIELDS:
            a, b = _bytes(getattr(g, f)), _bytes(getattr(w, f))
            assert (a is None) == (b is None), (i, f)
            if a is not None:
                assert np.array_equal(a, b), (i, f, int(np.count_nonzero(a != b)))
    return got


def test_group_mixed_shapes_and_roles():
    _group_vs_single([(384, 512), (1024, 256), (128, 128)], ["activation", "weight", "grad"],
                     sigmas=[1.0, 0.02, 1e-3])


def test_group_four_members():
    _group_vs_single([(256, 384), (128, 1024), (640, 128), (256, 256)],
                     ["activation", "weight", "weight", "grad"])


def test_group_bf16_column_copies():
    # --fp8-wgrad off: activation and gradient column copies are bf16 transposes, the weight's
    # stays FP8
    got = _group_vs_single([(256, 512), (512, 256), (384, 384)], ["activation", "weight", "grad"],
                           fp8_wgrad=False)
    assert [g.col_bf16 for g in got] == [1, 0, 1]


def test_group_with_empty_member():
    rec = F.Recipe(kind="mxfp8")
    x0 = to_dev_bf16(bf16_bits_normal(256, 256, seed=4, stream=20))
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    x2 = to_dev_bf16(bf16_bits_normal(128, 512, seed=4, stream=21))
    got = F.quantize_group(rec, [x0, e, x2], ["activation", "activation", "weight"])
    want = [F.quantize(rec, x0, "activation"), F.quantize(rec, x2, "weight")]
    torch.cuda.synchronize()
    assert (got[1].rows, got[1].cols) == (0, 256)
    for g, w in zip((got[0], got[2]), want):
        for f in FIELDS:
            assert np.array_equal(_bytes(getattr(g, f)), _bytes(getattr(w, f))), f


def test_group_against_oracle():
    shapes = [(256, 384), (128, 256)]
    bits = [bf16_bits_normal(r, c, seed=5, stream=30 + i, outlier_p=0.01)
            for i, (r, c) in enumerate(shapes)]
    rec = F.Recipe(kind="mxfp8")
    got = F.quantize_group(rec, [to_dev_bf16(b) for b in bits], ["activation", "weight"])
    torch.cuda.synchronize()
    for g, b in zip(got, bits):
        R, C = b.shape
        ref = O.quantize_mxfp8(b)
        assert np.array_equal(g.row.cpu().numpy(), ref["row"])
        assert np.array_equal(mx_untile(g.row_scale.cpu().numpy(), R, C), ref["row_scale"])
        assert np.array_equal(g.col.cpu().numpy(), ref["col"])
        assert np.array_equal(mx_untile(g.col_scale.cpu().numpy(), C, R), ref["col_scale"])


def test_group_mlp_step_tensors_full_size():
    # the benchmark's grouped launch: X 8192 x 4096, W1 16384 x 4096, W2 4096 x 16384
    _group_vs_single([(8192, 4096), (16384, 4096), (4096, 16384)],
                     ["activation", "weight", "weight"], sigmas=[1.0, 0.02, 0.02],
                     streams=[0, 1, 3])


def test_group_one_copy_only():
    # want_row = 0: only the column copies (and their scales) are written
    rec = F.Recipe(kind="mxfp8")
    xs = [to_dev_bf16(bf16_bits_normal(r, c, seed=6, stream=40 + i))
          for i, (r, c) in enumerate([(256, 512), (384, 128)])]
    roles = ["activation", "grad"]
    got = F.quantize_group(rec, xs, roles, want_row=False)
    want = [F.quantize(rec, x, r, want_row=False) for x, r in zip(xs, roles)]
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert g.row is None and w.row is None
        assert np.array_equal(_bytes(g.col), _bytes(w.col))
        assert np.array_equal(_bytes(g.col_scale), _bytes(w.col_scale))


@pytest.mark.parametrize("extra", [{}, {"format": "hybrid"}, {"power_2_scales": True},
                                   {"fp8_wgrad": False}, {"margin": 2}])
def test_group_blockwise(extra):
    # 1x128 activation and gradient blocks, 128x128 weight blocks, in one launch; under the
    # hybrid format the gradient's codes are E5M2
    rec = F.Recipe(kind="blockwise", **extra)
    shapes, roles = [(384, 512), (512, 256), (256, 384)], ["activation", "weight", "grad"]
    xs = [to_dev_bf16(bf16_bits_normal(r, c, seed=7, stream=50 + i, sigma=s, outlier_p=1e-2))
          for i, ((r, c), s) in enumerate(zip(shapes, [1.0, 0.02, 1e-3]))]
    got = F.quantize_group(rec, xs, roles)
    want = [F.quantize(rec, x, r) for x, r in zip(xs, roles)]
    torch.cuda.synchronize()
    for i, (g, w) in enumerate(zip(got, want)):
        assert (g.kind, g.role, g.col_bf16) == (w.kind, w.role, w.col_bf16), i
        for f in FIELDS:
            a, b = _bytes(getattr(g, f)), _bytes(getattr(w, f))
            assert (a is None) == (b is None), (i, f)
            if a is not None:
                assert np.array_equal(a, b), (i, f, int(np.count_nonzero(a != b)))


def test_group_blockwise_against_oracle():
    rec = F.Recipe(kind="blockwise")
    xb, wb = bf16_bits_normal(256, 384, seed=8, stream=60), bf16_bits_normal(384, 256, seed=8,
                                                                             stream=61, sigma=0.02)
    gx, gw = F.quantize_group(rec, [to_dev_bf16(xb), to_dev_bf16(wb)], ["activation", "weight"])
    torch.cuda.synchronize()
    rx, rw = O.quantize_blockwise_1x128(xb), O.quantize_blockwise_128x128(wb)
    assert np.array_equal(gx.row.cpu().numpy(), rx["row"])
    assert np.array_equal(gx.col.cpu().numpy(), rx["col"])
    assert np.array_equal(bw_untile(gx.row_scale.cpu().numpy(), 256, 384), rx["row_scale_inv"])
    assert np.array_equal(bw_untile(gx.col_scale.cpu().numpy(), 384, 256), rx["col_scale_inv"])
    assert np.array_equal(gw.row.cpu().numpy(), rw["row"])
    assert np.array_equal(gw.col.cpu().numpy(), rw["col"])
    assert np.array_equal(gw.row_scale.cpu().numpy(), rw["row_scale_inv"])
    assert np.array_equal(gw.col_scale.cpu().numpy(), rw["col_scale_inv"])
