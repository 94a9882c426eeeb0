"""GPU parity of the MXFP8 transformer MLP block (fc1 -> GeLU with its input kept in FP8 ->
fc2, then the backward pass) against the oracle, stage by stage and end to end.

Stage by stage: each GEMM's bf16 output against the oracle's fp64 sum (the GEMM tolerance);
the GeLU / dGeLU stage, given the GPU's own bf16 input, within one bf16 unit in the last place
of the oracle's fp64 evaluation (the GPU evaluates in fp32); and each quantisation exactly:
the oracle's MXFP8 quantiser applied to the GPU's bf16 quantiser input must give every code
and every E8M0 byte of both copies. End to end the GEMM outputs are compared with the oracle
run on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

from helpers import cuda_ok, from_dev_bf16, gemm_bf16_close, mx_untile, to_dev_bf16
from oracle import fp8_oracle as O
from workloads import bf16_bits_normal

pytestmark = pytest.mark.gpu

if cuda_ok():
    import scaled_quantize_fp8_gb300 as F


def _ulp_diff(a_bits, b_bits):
    """Distance in bf16 units in the last place (same-sign values)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def _mx_exact(gpu_q, gpu_in_bits, R, C):
    """Both copies of gpu_q equal the oracle's MXFP8 quantisation of the GPU's own bf16
    quantiser input, on every block."""
    ref = O.quantize_mxfp8(gpu_in_bits, want_col=gpu_q.col is not None)
    assert np.array_equal(gpu_q.row.cpu().numpy(), ref["row"])
    assert np.array_equal(mx_untile(gpu_q.row_scale.cpu().numpy(), R, C), ref["row_scale"])
    if gpu_q.col is not None:
        assert np.array_equal(gpu_q.col.cpu().numpy(), ref["col"])
        assert np.array_equal(mx_untile(gpu_q.col_scale.cpu().numpy(), C, R), ref["col_scale"])


@pytest.mark.parametrize("R,C", [(256, 384), (128, 1024)])
def test_gelu_quantize_stage(R, C):
    rec = F.Recipe(kind="mxfp8")
    hb = bf16_bits_normal(R, C, seed=41, sigma=2.0)
    a_q, h_q, a_bf16 = F.gelu_quantize(rec, to_dev_bf16(hb), want_a_bf16=True)
    torch.cuda.synchronize()
    # h's FP8 copy comes straight from the seeded input: bit-exact
    qh = O.quantize_mxfp8(hb, want_col=False)
    assert np.array_equal(h_q.row.cpu().numpy(), qh["row"])
    assert np.array_equal(mx_untile(h_q.row_scale.cpu().numpy(), R, C), qh["row_scale"])
    # a = gelu(h): one bf16 ulp at most; then a's codes and scales exactly
    a_ref = O.gelu_bf16(hb)
    a_gpu = from_dev_bf16(a_bf16)
    assert np.max(_ulp_diff(a_gpu, a_ref)) <= 1
    _mx_exact(a_q, a_gpu, R, C)


@pytest.mark.parametrize("R,C", [(256, 384), (128, 1024)])
def test_dgelu_quantize_stage(R, C):
    rec = F.Recipe(kind="mxfp8")
    hb = bf16_bits_normal(R, C, seed=42, sigma=2.0)
    dab = bf16_bits_normal(R, C, seed=43, sigma=1e-3)
    _, h_q, _ = F.gelu_quantize(rec, to_dev_bf16(hb))
    dh_q, dh_bf16 = F.dgelu_quantize(rec, to_dev_bf16(dab), h_q, want_dh_bf16=True)
    torch.cuda.synchronize()
    qh = O.quantize_mxfp8(hb, want_col=False)
    dh_ref = O.dgelu_bf16(dab, qh["row"], qh["row_scale"])
    dh_gpu = from_dev_bf16(dh_bf16)
    assert np.max(_ulp_diff(dh_gpu, dh_ref)) <= 1
    _mx_exact(dh_q, dh_gpu, R, C)


def _mlp(M, H, Fd, seed=0):
    rec = F.Recipe(kind="mxfp8")
    xb = bf16_bits_normal(M, H, seed=seed, stream=0)
    w1b = bf16_bits_normal(Fd, H, seed=seed, stream=1, sigma=0.02)
    w2b = bf16_bits_normal(H, Fd, seed=seed, stream=3, sigma=0.02)
    dyb = bf16_bits_normal(M, H, seed=seed, stream=2, sigma=1e-3)
    # GPU
    xq = F.quantize(rec, to_dev_bf16(xb), "activation")
    w1q = F.quantize(rec, to_dev_bf16(w1b), "weight")
    w2q = F.quantize(rec, to_dev_bf16(w2b), "weight")
    h = F.linear_fwd(rec, xq, w1q)
    a_q, h_q, a_bf16 = F.gelu_quantize(rec, h, want_a_bf16=True)
    y = F.linear_fwd(rec, a_q, w2q)
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    da, dw2 = F.linear_bwd(rec, dyq, a_q, w2q)
    dh_q, dh_bf16 = F.dgelu_quantize(rec, da, h_q, want_dh_bf16=True)
    dx, dw1 = F.linear_bwd(rec, dh_q, xq, w1q)
    torch.cuda.synchronize()
    # stage by stage on the GPU's own intermediates: GeLU / dGeLU within one ulp, then every
    # byte of the MXFP8 copies of h, a and dh
    h_g, a_g, da_g, dh_g = (from_dev_bf16(t) for t in (h, a_bf16, da, dh_bf16))
    assert np.max(_ulp_diff(a_g, O.gelu_bf16(h_g))) <= 1
    _mx_exact(h_q, h_g, M, Fd)
    _mx_exact(a_q, a_g, M, Fd)
    qh_g = O.quantize_mxfp8(h_g, want_col=False)
    assert np.max(_ulp_diff(dh_g, O.dgelu_bf16(da_g, qh_g["row"], qh_g["row_scale"]))) <= 1
    _mx_exact(dh_q, dh_g, M, Fd)
    # oracle, end to end from the same seeded inputs
    qx, qw1, qw2, qdy = (O.quantize_mxfp8(b) for b in (xb, w1b, w2b, dyb))
    dq = lambda q, c: O.dequant_mx(q[c], q[c + "_scale"])  # noqa: E731
    h_r = O.f64_to_bf16(O.gemm_tn_f64(dq(qx, "row"), dq(qw1, "row")))
    qh = O.quantize_mxfp8(h_r, want_col=False)
    a_r = O.gelu_bf16(h_r)
    qa = O.quantize_mxfp8(a_r)
    y_r = O.gemm_tn_f64(dq(qa, "row"), dq(qw2, "row"))
    da_r64 = O.gemm_tn_f64(dq(qdy, "row"), dq(qw2, "col"))
    dw2_r = O.gemm_tn_f64(dq(qdy, "col"), dq(qa, "col"))
    dh_r = O.dgelu_bf16(O.f64_to_bf16(da_r64), qh["row"], qh["row_scale"])
    qdh = O.quantize_mxfp8(dh_r)
    dx_r = O.gemm_tn_f64(dq(qdh, "row"), dq(qw1, "col"))
    dw1_r = O.gemm_tn_f64(dq(qdh, "col"), dq(qx, "col"))
    out = {}
    for name, got, ref in (("y", y, y_r), ("da", da, da_r64), ("dw2", dw2, dw2_r),
                           ("dx", dx, dx_r), ("dw1", dw1, dw1_r)):
        ok, err = gemm_bf16_close(from_dev_bf16(got), ref)
        out[name] = err
        assert ok, (name, err)
    return out


def test_mlp_block_small():
    _mlp(256, 256, 512)


def test_mlp_block_multi_tile():
    _mlp(384, 512, 1024, seed=1)


def _all_bf16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)


def _ulp_ok(gpu_bits, ref_bits):
    g = O.bf16_to_f32(gpu_bits)
    r = O.bf16_to_f32(ref_bits)
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan)
    return int(np.max(_ulp_diff(gpu_bits[~nan], ref_bits[~nan])))


def test_gelu_every_bf16_input():
    """a = gelu(h) for all 65,536 bf16 bit patterns (table range, tiny, huge, Inf, NaN)."""
    rec = F.Recipe(kind="mxfp8")
    hb = _all_bf16()
    _, _, a_bf16 = F.gelu_quantize(rec, to_dev_bf16(hb), want_a_bf16=True)
    torch.cuda.synchronize()
    assert _ulp_ok(from_dev_bf16(a_bf16), O.gelu_bf16(hb)) <= 1


def test_dgelu_every_bf16_input():
    """dh = 1 * gelu'(deq(h_fp8)) with h running over all 65,536 bf16 patterns."""
    rec = F.Recipe(kind="mxfp8")
    hb = _all_bf16()
    ones = np.full(hb.shape, 0x3F80, np.uint16)
    _, h_q, _ = F.gelu_quantize(rec, to_dev_bf16(hb))
    _, dh = F.dgelu_quantize(rec, to_dev_bf16(ones), h_q, want_dh_bf16=True)
    torch.cuda.synchronize()
    qh = O.quantize_mxfp8(hb, want_col=False)
    ref = O.dgelu_bf16(ones, qh["row"], qh["row_scale"])
    assert _ulp_ok(from_dev_bf16(dh), ref) <= 1
