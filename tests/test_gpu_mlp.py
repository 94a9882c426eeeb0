"""GPU parity of the MXFP8 transformer MLP block (fc1 -> GeLU with its input kept in FP8 ->
fc2, then the backward pass) against the oracle run end to end on the same seeded inputs.

GeLU is computed in fp32 on the GPU and in float64 by the oracle, so the bf16 activations may
differ by one unit in the last place; where a whole 1x32 block of the activation agrees
bit-exactly its FP8 codes and scale must agree bit-exactly, elsewhere codes may differ by one
step. GEMM outputs are compared within the GEMM tolerance.
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


def _mx_codes_agree_where_inputs_agree(gpu_q, gpu_in_bits, ref_in_bits, R, C):
    """Row copy: blocks (1x32 along C) whose inputs agree exactly must agree exactly."""
    ref = O.quantize_mxfp8(ref_in_bits)
    same = (gpu_in_bits == ref_in_bits).reshape(R, C // 32, 32).all(axis=2)
    rows = gpu_q.row.cpu().numpy().reshape(R, C // 32, 32)
    assert np.array_equal(rows[same], ref["row"].reshape(R, C // 32, 32)[same])
    sc = mx_untile(gpu_q.row_scale.cpu().numpy(), R, C)
    assert np.array_equal(sc[same], ref["row_scale"][same])
    # blocks whose inputs differ by an ulp: dequantised values stay within two E4M3 steps
    dg = O.e4m3_decode(rows) * O.e8m0_decode(sc)[:, :, None]
    dr = O.e4m3_decode(ref["row"].reshape(R, C // 32, 32)) * O.e8m0_decode(ref["row_scale"])[:, :, None]
    tol = 0.25 * np.abs(dr) + 2.0 ** -9 * O.e8m0_decode(ref["row_scale"])[:, :, None]
    assert np.all(np.abs(dg - dr)[~same] <= tol[~same])
    return same.mean()


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
    # a = gelu(h): one bf16 ulp at most
    a_ref = O.gelu_bf16(hb)
    a_gpu = from_dev_bf16(a_bf16)
    assert np.max(_ulp_diff(a_gpu, a_ref)) <= 1
    frac = _mx_codes_agree_where_inputs_agree(a_q, a_gpu, a_ref, R, C)
    assert frac > 0.5


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
    _mx_codes_agree_where_inputs_agree(dh_q, dh_gpu, dh_ref, R, C)


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
    a_q, h_q, _ = F.gelu_quantize(rec, h)
    y = F.linear_fwd(rec, a_q, w2q)
    dyq = F.quantize(rec, to_dev_bf16(dyb), "grad")
    da, dw2 = F.linear_bwd(rec, dyq, a_q, w2q)
    dh_q, _ = F.dgelu_quantize(rec, da, h_q)
    dx, dw1 = F.linear_bwd(rec, dh_q, xq, w1q)
    torch.cuda.synchronize()
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
