"""Pins for the oracle's dequantise-then-matmul GEMMs and the GeLU stage.

GEMMs are checked against exact rational arithmetic (fractions.Fraction, pure-Python loops on
tiny inputs: 8x8 tensorwise, 8x32 MXFP8, 8x128 blockwise), against identity operands, and
against the dequantised operands for transposed roles. GeLU is pinned to tabulated values of
the standard normal CDF, to its limits and to finite differences.
"""
import math
from fractions import Fraction

import numpy as np

from oracle import fp8_oracle as O
from workloads import bf16_bits_from_f32, bf16_bits_normal


def _frac_decode(code):
    code = int(code)
    e, m = (code >> 3) & 0xF, code & 7
    v = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if code & 0x80 else v


def _exact_tn(A, B):
    """sum_k A[m][k] * B[n][k] over Fractions."""
    return [[sum(a * b for a, b in zip(ra, rb)) for rb in B] for ra in A]


def _close(c64, exact, rel=1e-12):
    scale = max(abs(float(v)) for row in exact for v in row) or 1.0
    for i, row in enumerate(exact):
        for j, v in enumerate(row):
            assert abs(c64[i, j] - float(v)) <= rel * scale, (i, j, c64[i, j], float(v))


def test_tensorwise_8x8_exact():
    x = bf16_bits_normal(8, 8, seed=21)
    w = bf16_bits_normal(8, 8, seed=22, sigma=0.02)
    qx, qw = O.quantize_tensorwise(x), O.quantize_tensorwise(w)
    c = O.gemm_tn_f64(O.dequant_tensor(qx["row"], qx["scale_inv"]),
                      O.dequant_tensor(qw["row"], qw["scale_inv"]))
    sx, sw = Fraction(float(qx["scale_inv"])), Fraction(float(qw["scale_inv"]))
    A = [[_frac_decode(v) * sx for v in r] for r in qx["row"]]
    B = [[_frac_decode(v) * sw for v in r] for r in qw["row"]]
    _close(c, _exact_tn(A, B))


def test_mx_8x32_exact():
    x = bf16_bits_normal(32, 32, seed=23, outlier_p=0.05)
    w = bf16_bits_normal(32, 32, seed=24, sigma=0.02)
    qx, qw = O.quantize_mxfp8(x), O.quantize_mxfp8(w)
    c = O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]),
                      O.dequant_mx(qw["row"], qw["row_scale"]))[:8, :8]
    A = [[_frac_decode(v) * Fraction(2) ** (int(qx["row_scale"][i, 0]) - 127)
          for v in qx["row"][i]] for i in range(8)]
    B = [[_frac_decode(v) * Fraction(2) ** (int(qw["row_scale"][j, 0]) - 127)
          for v in qw["row"][j]] for j in range(8)]
    _close(c, _exact_tn(A, B))


def test_blockwise_8x128_exact():
    x = bf16_bits_normal(128, 128, seed=25)
    w = bf16_bits_normal(128, 128, seed=26, sigma=0.02)
    qx = O.quantize_blockwise_1x128(x)
    qw = O.quantize_blockwise_128x128(w)
    c = O.gemm_tn_f64(O.dequant_1x128(qx["row"], qx["row_scale_inv"]),
                      O.dequant_128x128(qw["row"], qw["row_scale_inv"]))[:8, :8]
    A = [[_frac_decode(v) * Fraction(float(qx["row_scale_inv"][i, 0])) for v in qx["row"][i]]
         for i in range(8)]
    sw = Fraction(float(qw["row_scale_inv"][0, 0]))
    B = [[_frac_decode(v) * sw for v in qw["row"][j]] for j in range(8)]
    _close(c, _exact_tn(A, B))


def test_identity_weight_reproduces_dequantised_x():
    x = bf16_bits_normal(64, 64, seed=27)
    qx = O.quantize_tensorwise(x)
    eye = bf16_bits_from_f32(np.eye(64, dtype=np.float32))
    qi = O.quantize_tensorwise(eye)
    y = O.gemm_tn_f64(O.dequant_tensor(qx["row"], qx["scale_inv"]),
                      O.dequant_tensor(qi["row"], qi["scale_inv"]))
    assert np.array_equal(y, O.dequant_tensor(qx["row"], qx["scale_inv"]) *
                          float(qi["scale_inv"]) * 448.0)


def test_gemm_roles_transpose_consistently():
    # wgrad from the column-wise copies equals the transpose-contracted row-wise math when the
    # copies are byte transposes (tensorwise): dW = dY^T X
    dy = bf16_bits_normal(32, 16, seed=28, sigma=1e-3)
    x = bf16_bits_normal(32, 24, seed=29)
    qd, qx = O.quantize_tensorwise(dy), O.quantize_tensorwise(x)
    dw = O.gemm_tn_f64(O.dequant_tensor(qd["col"], qd["scale_inv"]),
                       O.dequant_tensor(qx["col"], qx["scale_inv"]))
    ref = (O.dequant_tensor(qd["row"], qd["scale_inv"]).T
           @ O.dequant_tensor(qx["row"], qx["scale_inv"]))
    assert np.max(np.abs(dw - ref)) <= 1e-13 * np.max(np.abs(ref))


def test_bf16_result_rounding_within_half_ulp():
    x = bf16_bits_normal(16, 64, seed=30)
    w = bf16_bits_normal(16, 64, seed=31)
    r = O.bf16_gemm_tn_f64(x, w)
    rb = O.bf16_to_f32(O.f64_to_bf16(r)).astype(np.float64)
    assert np.all(np.abs(rb - r) <= np.abs(r) * 2.0 ** -8 + 1e-300)


def test_gelu_tabulated_normal_cdf():
    # Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208 (standard normal tables)
    assert abs(O.gelu_f64(1.0) - 0.8413447460685429) < 1e-15
    assert abs(O.gelu_f64(-1.0) + (1 - 0.8413447460685429)) < 1e-15
    assert abs(O.gelu_f64(2.0) - 2 * 0.9772498680518208) < 1e-15
    assert O.gelu_f64(0.0) == 0.0
    assert abs(O.gelu_f64(12.0) - 12.0) < 1e-12
    assert abs(O.gelu_f64(-12.0)) < 1e-12
    # gelu'(0) = 1/2; phi(1) = 0.24197072451914337
    assert abs(O.gelu_grad_f64(0.0) - 0.5) < 1e-15
    assert abs(O.gelu_grad_f64(1.0) - (0.8413447460685429 + 0.24197072451914337)) < 1e-15


def test_gelu_negative_tail_keeps_relative_precision():
    # Phi(-8) = 6.220960574271784e-16, Phi(-10) = 7.61985302416047e-24 (standard normal tables)
    assert abs(O.gelu_f64(-8.0) / (-8.0 * 6.220960574271784e-16) - 1) < 1e-12
    assert abs(O.gelu_f64(-10.0) / (-10.0 * 7.61985302416047e-24) - 1) < 1e-12
    # phi(-8) = 5.052271083536893e-15: gelu'(-8) = Phi(-8) - 8 phi(-8)
    assert abs(O.gelu_grad_f64(-8.0) / (6.220960574271784e-16 - 8 * 5.052271083536893e-15) - 1) < 1e-12


def test_gelu_grad_matches_finite_difference():
    h = np.linspace(-6, 6, 241)
    eps = 1e-6
    fd = (O.gelu_f64(h + eps) - O.gelu_f64(h - eps)) / (2 * eps)
    assert np.max(np.abs(fd - O.gelu_grad_f64(h))) < 1e-8


def test_dgelu_reads_h_from_fp8_copy():
    h = bf16_bits_normal(32, 64, seed=32)
    da = bf16_bits_normal(32, 64, seed=33, sigma=1e-3)
    qh = O.quantize_mxfp8(h)
    dh = O.dgelu_bf16(da, qh["row"], qh["row_scale"])
    hq = O.dequant_mx(qh["row"], qh["row_scale"])
    ref = O.bf16_to_f32(da).astype(np.float64) * np.array(
        [0.5 * math.erfc(-v / math.sqrt(2)) + v * math.exp(-v * v / 2) / math.sqrt(2 * math.pi)
         for v in hq.ravel()]).reshape(hq.shape)
    assert np.array_equal(dh, O.f64_to_bf16(ref))


def _frac_decode_e5m2(code):
    code = int(code)
    e, m = (code >> 2) & 0x1F, code & 3
    v = Fraction(m, 65536) if e == 0 else (1 + Fraction(m, 4)) * Fraction(2) ** (e - 15)
    return -v if code & 0x80 else v


def test_hybrid_dgrad_8x8_exact():
    """Hybrid format: an E5M2 gradient times an E4M3 weight (dgrad), decoded by hand."""
    dy = bf16_bits_normal(8, 8, seed=25, sigma=1e-3)
    w = bf16_bits_normal(8, 8, seed=26, sigma=0.02)
    qd, qw = O.quantize_tensorwise(dy, fmt="e5m2"), O.quantize_tensorwise(w)
    c = O.gemm_tn_f64(O.dequant_tensor(qd["row"], qd["scale_inv"], fmt="e5m2"),
                      O.dequant_tensor(qw["col"], qw["scale_inv"]))
    sd, sw = Fraction(float(qd["scale_inv"])), Fraction(float(qw["scale_inv"]))
    A = [[_frac_decode_e5m2(v) * sd for v in r] for r in qd["row"]]
    B = [[_frac_decode(v) * sw for v in r] for r in qw["col"]]
    _close(c, _exact_tn(A, B))
