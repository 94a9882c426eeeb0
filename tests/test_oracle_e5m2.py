"""Pins for the oracle's E5M2 encoding (the gradient format of the hybrid recipe) and the
hybrid scale rule, against facts outside the oracle.

Pins used: the format's fixed values (tests/golden/e5m2_facts.txt), torch's float8_e5m2
conversion (an independent library routine), brute force over the finite E5M2 values for
every bf16 bit pattern, and the scale's defining property (the amax element lands on the
format's largest value).
"""
import math
import os

import numpy as np
import torch

from oracle import fp8_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_table():
    """The 124 non-negative finite E5M2 magnitudes (codes 0x00..0x7B) from the bit fields."""
    vals = []
    for code in range(0x7C):
        e, m = code >> 2, code & 3
        vals.append(m * 2.0 ** -16 if e == 0 else (1 + m / 4) * 2.0 ** (e - 15))
    return np.array(vals)


def _brute_encode(v):
    """Nearest finite magnitude (ties to the even code), saturate at 57344, keep the sign."""
    table = _finite_table()
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    idx_hi = np.clip(np.searchsorted(table, a), 1, len(table) - 1)
    lo, hi = table[idx_hi - 1], table[idx_hi]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (idx_hi % 2 == 0))
    out = np.where(pick_hi, idx_hi, idx_hi - 1)
    out = np.where(a >= 57344.0, 0x7B, out)
    out = np.where(a <= 0.0, 0, out)
    out = np.where(np.isnan(v), 0x7F, out)
    return (out | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_golden_facts():
    n = 0
    for line in open(os.path.join(GOLDEN, "e5m2_facts.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        tok = line.split()
        v, want = float(tok[0]), int(tok[1], 16)
        got = int(O.e5m2_encode(np.float32(v)))
        if math.isnan(v):
            assert got & 0x7F == 0x7F
        else:
            assert got == want, (v, hex(got), hex(want))
        n += 1
    assert n >= 18


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e5m2_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])            # includes +-inf at 0x7C / 0xFC
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert O.e5m2_decode(np.uint8(0x7B)) == 57344.0 and O.e5m2_decode(np.uint8(0x01)) == 2.0 ** -16


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], dtype=np.uint8)
    assert len(codes) == 248
    back = O.e5m2_encode(O.e5m2_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_encode_all_bf16_against_brute_force():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = O.bf16_to_f32(bits)
    for s in (1.0, 3.0, 2.0 ** -10, 2.0 ** 12, 0.3):
        v = (x * np.float32(s)).astype(np.float32)
        got = O.e5m2_encode(v)
        want = _brute_encode(v.astype(np.float64))
        nan = np.isnan(v)
        assert np.array_equal(got[~nan], want[~nan]), s
        assert np.all(got[nan] & 0x7F == 0x7F)


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(1 << 20) * np.exp(rng.uniform(-12, 10, 1 << 20))).astype(np.float32)
    v = v[np.abs(v) < 57344.0]
    ref = torch.from_numpy(v).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(O.e5m2_encode(v), ref)


def test_hybrid_scale_maps_amax_to_57344():
    rng = np.random.default_rng(6)
    x = O.f64_to_bf16(rng.standard_normal((64, 128)) * 1e-3)
    q = O.quantize_tensorwise(x, fmt="e5m2")
    i = np.unravel_index(np.argmax(np.abs(O.bf16_to_f32(x))), x.shape)
    assert O.e5m2_decode(q["row"][i]) in (57344.0, -57344.0)
    assert np.float32(q["scale"]) == np.float32(np.float32(57344.0) / q["amax"])
    # the same tensor under E4M3 keeps the 448 rule
    assert O.e4m3_decode(O.quantize_tensorwise(x)["row"][i]) in (448.0, -448.0)
    assert O.hybrid_format("grad") == "e5m2" and O.hybrid_format("activation") == "e4m3"


def test_hybrid_blockwise_and_delayed():
    rng = np.random.default_rng(7)
    x = O.f64_to_bf16(rng.standard_normal((128, 256)))
    q = O.quantize_blockwise_1x128(x, fmt="e5m2")
    deq = O.dequant_1x128(q["row"], q["row_scale_inv"], fmt="e5m2")
    xf = O.bf16_to_f32(x).astype(np.float64)
    # E5M2 keeps 2 mantissa bits: relative error at most 2^-3 above the block's subnormals
    big = np.abs(xf) > np.repeat(np.max(np.abs(xf).reshape(128, 2, 128), axis=2), 128, 1) * 2.0 ** -12
    assert np.all(np.abs(deq - xf)[big] <= np.abs(xf)[big] * 2.0 ** -3)
    d = O.DelayedScaling(4, fmt="e5m2")
    d.quantize(x)
    s, _ = d.update(np.float32(2.0))
    assert s == np.float32(57344.0 / 2.0)
