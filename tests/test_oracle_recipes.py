"""Pins for the oracle's recipe arithmetic: tensorwise / delayed / MXFP8 / blockwise scales.

Each test checks a fact that does not come from re-running the oracle's own formula: hand
values (tests/golden/*.txt), brute-force searches over the definition, invariants under
power-of-two rescaling, and reductions of one recipe to another on special inputs.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp8_oracle as O
from workloads import bf16_bits_from_f32, bf16_bits_normal

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    for line in open(os.path.join(GOLDEN, name)):
        if line.strip() and not line.startswith("#"):
            yield line.split()


# ---------------------------------------------------------------- tensorwise scale

def test_scale_fixed_values():
    s, si = O.scale_from_amax(448.0)
    assert s == 1.0 and si == 1.0
    s, si = O.scale_from_amax(1.0)
    assert s == 448.0 and si == np.float32(1.0) / np.float32(448.0)
    s, si = O.scale_from_amax(2.0, margin=3)
    assert s == 28.0                                   # 224 * 2^-3
    for bad in (0.0, np.inf, np.nan):
        assert O.scale_from_amax(bad) == (1.0, 1.0)
    s, _ = O.scale_from_amax(1e-41)                    # 448 / tiny overflows fp32
    assert s == np.finfo(np.float32).max
    # 448/3 in fp32 is the float nearest to the rational 448/3
    s, _ = O.scale_from_amax(3.0)
    assert abs(Fraction(float(s)) - Fraction(448, 3)) <= Fraction(float(np.spacing(s))) / 2


def test_margin_is_exact_power_of_two():
    for amax in (0.37, 1.0, 5.5, 1234.0):
        s0, _ = O.scale_from_amax(amax, 0)
        for m in range(0, 8):
            sm, _ = O.scale_from_amax(amax, m)
            assert Fraction(float(sm)) == Fraction(float(s0)) / 2 ** m


def test_tensorwise_amax_element_hits_448_and_transpose():
    x = bf16_bits_normal(64, 96, seed=5)
    q = O.quantize_tensorwise(x)
    xf = O.bf16_to_f32(x)
    i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert q["row"][i] in (0x7E, 0xFE)
    assert np.array_equal(q["col"], q["row"].T)
    dq = O.e4m3_decode(q["row"])
    assert np.all(np.abs(dq) <= 448.0)


def test_tensorwise_invariant_under_power_of_two_rescale():
    x = bf16_bits_normal(32, 64, seed=6)
    xf = O.bf16_to_f32(x)
    q0 = O.quantize_tensorwise(x)
    for k in (-20, -3, 5, 40):
        xk = O.bf16_to_f32(bf16_bits_from_f32(np.ldexp(xf, k)))
        assert np.array_equal(np.ldexp(xf, k), xk)   # the rescale is exact
        qk = O.quantize_tensorwise(bf16_bits_from_f32(xk))
        assert np.array_equal(qk["row"], q0["row"])
        assert Fraction(float(qk["scale"])) == Fraction(float(q0["scale"])) / Fraction(2) ** k


def test_tensorwise_codes_are_nearest_to_scaled_value():
    x = bf16_bits_normal(16, 32, seed=8)
    q = O.quantize_tensorwise(x, margin=1)
    xf = O.bf16_to_f32(x).astype(np.float64)
    scaled = (xf * float(q["scale"]))
    dq = O.e4m3_decode(q["row"])
    # every code is within half an E4M3 step of the scaled value (no saturation with margin 1)
    finite = np.sort(np.unique(np.abs(O.e4m3_decode(np.arange(0x7F, dtype=np.uint8)))))
    step = np.array([finite[np.searchsorted(finite, abs(d))+1] - abs(d) if abs(d) < 448 else 32
                     for d in dq.ravel()]).reshape(dq.shape)
    assert np.all(np.abs(dq - scaled) <= step / 2 * (1 + 1e-9) + 2.0 ** -10)


# ---------------------------------------------------------------- delayed

def test_delayed_scripted_sequence():
    hdr = [l for l in open(os.path.join(GOLDEN, "delayed_sequence.txt")) if l.startswith("# ")]
    L = int([h for h in hdr if h.startswith("# history_len")][0].split()[2])
    amaxes = [float(t) for t in [h for h in hdr if h.startswith("# amax ")][0].split()[2:]]
    want = {int(t[0]): Fraction(t[1]) for t in _lines("delayed_sequence.txt")}
    d = O.DelayedScaling(L)
    got = [d.scale]
    for a in amaxes:
        d.update(a)
        got.append(d.scale)
    for step, w in want.items():
        s = got[step]
        # fp32 of the rational value, correctly rounded
        assert abs(Fraction(float(s)) - w) <= Fraction(float(np.spacing(np.float32(s)))) / 2
        assert d.history.dtype == np.float32


def test_delayed_scripted_sequence_most_recent():
    hdr = [l for l in open(os.path.join(GOLDEN, "delayed_sequence_most_recent.txt"))
           if l.startswith("# ")]
    L = int([h for h in hdr if h.startswith("# history_len")][0].split()[2])
    amaxes = [float(t) for t in [h for h in hdr if h.startswith("# amax ")][0].split()[2:]]
    want = {int(t[0]): Fraction(t[1]) for t in _lines("delayed_sequence_most_recent.txt")}
    d = O.DelayedScaling(L, algo="most_recent")
    got = [d.scale]
    for a in amaxes:
        d.update(a)
        got.append(d.scale)
    for step, w in want.items():
        s = got[step]
        # fp32 of the rational value, correctly rounded
        assert abs(Fraction(float(s)) - w) <= Fraction(float(np.spacing(np.float32(s)))) / 2
    assert list(d.history) == [np.float32(0.25), np.float32(0.125), 2.0, 0.5]   # still recorded


def test_delayed_quantizes_with_previous_scale_and_saturates():
    d = O.DelayedScaling(8)
    x0 = bf16_bits_from_f32(np.full((4, 32), 2.0, np.float32))
    q0 = d.quantize(x0)
    assert q0["scale"] == 1.0 and np.all(q0["row"] == O.e4m3_encode(np.float32(2.0)))
    d.update(q0["amax"])                                # next scale 224
    x1 = bf16_bits_from_f32(np.full((4, 32), 4.0, np.float32))
    q1 = d.quantize(x1)
    assert q1["scale"] == 224.0
    assert np.all(q1["row"] == 0x7E)                    # 4 * 224 = 896 saturates to 448


def test_delayed_history_rejects_zero_length():
    with pytest.raises(ValueError):
        O.DelayedScaling(0)


# ---------------------------------------------------------------- MXFP8

def test_e8m0_golden_blocks():
    for tok in _lines("e8m0_blocks.txt"):
        amax, e, byte = float(tok[0]), int(tok[1]), int(tok[2])
        blk = np.zeros((1, 32), np.float32)
        blk[0, 5] = amax
        blk[0, 9] = -amax / 4
        q = O.quantize_mxfp8(bf16_bits_from_f32(np.repeat(blk, 32, axis=0)))
        amax_bf16 = O.bf16_to_f32(bf16_bits_from_f32(np.array([amax], np.float32)))
        assert int(O.mx_exponent(amax_bf16)[0]) == e
        assert q["row_scale"][0, 0] == byte, (amax, q["row_scale"][0, 0], byte)


def test_e8m0_is_smallest_covering_power_brute_force():
    g = np.random.default_rng(11)
    a = np.abs(O.bf16_to_f32(bf16_bits_from_f32(
        (g.standard_normal(4000) * np.exp(g.uniform(-60, 60, 4000))).astype(np.float32))))
    a = a[a >= 2.0 ** -126]
    e = O.mx_exponent(a)
    for ai, ei in zip(a.tolist(), e.tolist()):
        # search the definition directly over all candidate exponents
        best = next(k for k in range(-127, 128) if Fraction(ai) <= 448 * Fraction(2) ** k)
        assert ei == best


def test_mx_no_element_saturates_and_scaling_invariance():
    x = bf16_bits_normal(64, 128, seed=12, outlier_p=0.05)
    q = O.quantize_mxfp8(x)
    xf = O.bf16_to_f32(x).astype(np.float64)
    f = np.repeat(O.e8m0_decode(q["row_scale"]), 32, axis=1)
    assert np.all(np.abs(xf / f) <= 448.0)
    for k in (-9, 4):
        qk = O.quantize_mxfp8(bf16_bits_from_f32(np.ldexp(xf, k).astype(np.float32)))
        assert np.array_equal(qk["row"], q["row"])
        assert np.array_equal(qk["row_scale"].astype(int), q["row_scale"].astype(int) + k)
    # the column-wise copy is the row-wise recipe applied to X^T
    qt = O.quantize_mxfp8(np.ascontiguousarray(x.T))
    assert np.array_equal(qt["row"], q["col"]) and np.array_equal(qt["row_scale"], q["col_scale"])


def test_mx_floor_rule_would_saturate_ceil_rule_does_not():
    # amax with mantissa in (1.75, 2): the ceil rule must go one exponent up
    blk = np.zeros((32, 32), np.float32)
    blk[:, 0] = 1.875
    q = O.quantize_mxfp8(bf16_bits_from_f32(blk))
    assert np.all(q["row_scale"] == 120)                # e = -7: 1.875 * 128 = 240
    assert np.all(q["row"][:, 0] == 0x77)               # 240 exactly, not saturated


# ---------------------------------------------------------------- blockwise

def test_blockwise_1x128_uniform_blocks_reduce_to_tensorwise():
    # every 1x128 block holds the same amax -> every block scale equals the tensor scale
    x = O.bf16_to_f32(bf16_bits_normal(128, 256, seed=13))
    x = np.clip(x, -3.0, 3.0)
    x[:, ::128] = 3.0
    x[::128, :] = 3.0
    xb = bf16_bits_from_f32(x)
    t = O.quantize_tensorwise(xb, margin=2)
    b = O.quantize_blockwise_1x128(xb, margin=2)
    assert np.array_equal(b["row"], t["row"])
    assert np.array_equal(b["col"], t["col"])
    assert np.all(b["row_scale_inv"] == t["scale_inv"])
    assert np.all(b["col_scale_inv"] == t["scale_inv"])


def test_blockwise_128x128_tiles_independent_and_power_of_two_invariant():
    base = O.bf16_to_f32(bf16_bits_normal(128, 128, seed=14, sigma=0.02))
    ks = [[0, 3], [-5, 7]]
    full = np.block([[np.ldexp(base, ks[i][j]) for j in range(2)] for i in range(2)])
    q = O.quantize_blockwise_128x128(bf16_bits_from_f32(full))
    t0 = q["row"][:128, :128]
    for i in range(2):
        for j in range(2):
            assert np.array_equal(q["row"][128*i:128*i+128, 128*j:128*j+128], t0)
            assert (Fraction(float(q["row_scale_inv"][i, j]))
                    == Fraction(float(q["row_scale_inv"][0, 0])) * Fraction(2) ** ks[i][j])
    assert np.array_equal(q["col"], q["row"].T)
    assert np.array_equal(q["col_scale_inv"], q["row_scale_inv"].T)


def test_blockwise_each_block_max_hits_448():
    x = bf16_bits_normal(128, 384, seed=15)
    q = O.quantize_blockwise_1x128(x)
    xf = O.bf16_to_f32(x)
    for r in range(0, 128, 17):
        for j in range(3):
            blk = xf[r, 128*j:128*j+128]
            c = np.argmax(np.abs(blk))
            assert q["row"][r, 128*j + c] in (0x7E, 0xFE)


def test_mx_nonfinite_block_gets_nan_scale():
    blk = np.ones((32, 64), np.float32)
    blk[3, 40] = np.inf
    blk[7, 2] = np.nan
    q = O.quantize_mxfp8(bf16_bits_from_f32(blk))
    assert q["row_scale"][3, 1] == 255 and q["row_scale"][7, 0] == 255
    assert q["row_scale"][3, 0] == 119 and q["row_scale"][0, 1] == 119     # e = -8 for amax 1
    assert q["row"][3, 40] == 0x7E and (q["row"][7, 2] & 0x7F) == 0x7F
    assert q["row"][3, 41] == O.e4m3_encode(np.float32(1.0))                 # e = 0 in the NaN block
    assert np.isnan(O.e8m0_decode(np.uint8(255)))


def test_power_of_two_block_scales():
    """pow2 block scales are the largest power of two not above 448/amax: checked by brute
    search over the exponent, with the no-saturation property and exact s_inv."""
    rng = np.random.default_rng(11)
    amax = np.float32(np.exp(rng.uniform(-30, 30, 2000))).astype(np.float32)
    s, s_inv = O.scales_from_amax(amax, pow2=True)
    for a, v in zip(amax[:200], s[:200]):
        q = np.float32(np.float32(448.0) / a)
        k = max(e for e in range(-149, 128) if 2.0 ** e <= float(q))
        assert float(v) == 2.0 ** k
    assert np.all(s.astype(np.float64) * amax.astype(np.float64) <= 448.0)
    assert np.all(s.astype(np.float64) * s_inv.astype(np.float64) == 1.0)
    # margin: one more halving per bit
    s2, _ = O.scales_from_amax(amax, margin=2, pow2=True)
    assert np.array_equal(s2, (s / 4).astype(np.float32))
    x = bf16_bits_from_f32(rng.standard_normal((128, 256)).astype(np.float32))
    q = O.quantize_blockwise_1x128(x, pow2=True)
    f, _ = np.frexp(q["row_scale_inv"].astype(np.float64))
    assert np.all(f == 0.5)                                   # every s_inv a power of two


def test_fp32_master_weight_inputs():
    """Quantising fp32 master weights: fp32 values that bf16 holds exactly give the bf16
    path's bytes; other fp32 values are cast without a bf16 rounding (codes follow the fp32
    product), and the MX exponent is the smallest e with amax <= 448 * 2^e by brute search."""
    rng = np.random.default_rng(12)
    w32 = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    wb = O.f64_to_bf16(w32.astype(np.float64))
    w_exact = O.bf16_to_f32(wb)                               # fp32 copies of the bf16 values
    for f in (lambda x: O.quantize_tensorwise(x), lambda x: O.quantize_mxfp8(x),
              lambda x: O.quantize_blockwise_128x128(x)):
        a, b = f(wb), f(w_exact)
        for k in a:
            assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
    q = O.quantize_tensorwise(w32)
    s = np.float32(np.float32(448.0) / np.max(np.abs(w32)))
    assert q["scale"] == s
    assert np.array_equal(q["row"], O.e4m3_encode((w32 * s).astype(np.float32)))
    assert not np.array_equal(q["row"], O.quantize_tensorwise(wb)["row"])
    mx = O.quantize_mxfp8(w32, want_col=False)
    amax = np.max(np.abs(w32.reshape(256, 8, 32)), axis=2)
    for i in range(0, 256, 37):
        for j in range(8):
            e = min(k for k in range(-127, 128) if float(amax[i, j]) <= 448.0 * 2.0 ** k)
            assert mx["row_scale"][i, j] == e + 127


def test_pow2_scales_as_e8m0_dequantise_identically():
    """The E8M0 view of power-of-two block scales dequantises every code exactly as the fp32
    s_inv does (1x128 activations and 128x128 weights, both copies)."""
    rng = np.random.default_rng(13)
    x = bf16_bits_from_f32((rng.standard_normal((256, 384)) *
                            np.exp(rng.uniform(-6, 6, (256, 1)))).astype(np.float32))
    q = O.quantize_blockwise_1x128(x, pow2=True)
    b = O.pow2_scales_as_e8m0(q["row_scale_inv"], 1, 256, 384)
    assert np.array_equal(O.dequant_mx(q["row"], b), O.dequant_1x128(q["row"], q["row_scale_inv"]))
    bc = O.pow2_scales_as_e8m0(q["col_scale_inv"], 1, 384, 256)
    assert np.array_equal(O.dequant_mx(q["col"], bc), O.dequant_1x128(q["col"], q["col_scale_inv"]))
    w = O.quantize_blockwise_128x128(x, pow2=True)
    bw = O.pow2_scales_as_e8m0(w["row_scale_inv"], 128, 256, 384)
    assert np.array_equal(O.dequant_mx(w["row"], bw), O.dequant_128x128(w["row"], w["row_scale_inv"]))
    assert np.all(O.e8m0_decode(b) == np.repeat(q["row_scale_inv"], 4, axis=1))
