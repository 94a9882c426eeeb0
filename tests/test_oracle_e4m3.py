"""Pins for the oracle's E4M3 / bf16 / E8M0 encodings against facts outside the oracle.

Pins used: the format's fixed values (tests/golden/e4m3_facts.txt), torch's own float8_e4m3fn
and float8_e8m0fnu conversions (an independent library routine), and brute force over the
254 finite E4M3 values for every bf16 bit pattern.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import fp8_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_table():
    """The 127 non-negative finite E4M3 magnitudes, by brute decoding of the bit fields."""
    vals = []
    for code in range(0x7F):          # 0x00 .. 0x7E
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def _brute_encode(v):
    """Nearest finite magnitude (ties to the even code), saturate at 448, keep the sign."""
    table = _finite_table()
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    out = np.empty(v.shape, dtype=np.int64)
    idx_hi = np.clip(np.searchsorted(table, a), 1, len(table) - 1)
    lo, hi = table[idx_hi - 1], table[idx_hi]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (idx_hi % 2 == 0))
    out[:] = np.where(pick_hi, idx_hi, idx_hi - 1)
    out = np.where(a >= 448.0, 0x7E, out)
    out = np.where(a <= 0.0, 0, out)
    out = np.where(np.isnan(v), 0x7F, out)            # NaN keeps its sign bit as well
    return (out | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_golden_facts():
    path = os.path.join(GOLDEN, "e4m3_facts.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        tok = line.split()
        v = float(tok[0])
        want = int(tok[1], 16)
        got = int(O.e4m3_encode(np.float32(v)))
        if math.isnan(v):
            assert got & 0x7F == 0x7F
        else:
            assert got == want, (v, hex(got), hex(want))
        n += 1
    assert n >= 15


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert len(codes) == 254
    back = O.e4m3_encode(O.e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_decode_monotone():
    table = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(table) > 0)


@pytest.mark.parametrize("scale", [1.0, 448.0, 2.0 ** -7, 3.0, 1.0 / 3.0, 1e-30, 1e30])
def test_encode_exhaustive_bf16_vs_brute_force(scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = O.bf16_to_f32(bits)
    with np.errstate(over="ignore", invalid="ignore"):
        v = (x * np.float32(scale)).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(v), _brute_encode(v))


def test_encode_exhaustive_bf16_vs_torch_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = O.bf16_to_f32(bits)
    keep = np.isfinite(x) & (np.abs(x) < 464.0)      # torch's cast does not saturate
    ref = torch.from_numpy(x[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x[keep]), ref)


def test_encode_random_f32_vs_torch():
    g = np.random.default_rng(7)
    bits = g.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) < 464.0)
    ref = torch.from_numpy(x[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x[keep]), ref)


def test_bf16_rounding_vs_torch_and_single_rounding():
    g = np.random.default_rng(3)
    x = g.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), ref)
    # A float64 just above a bf16 tie must round up; rounding through float32 first would
    # land on the tie and pick the even neighbour 1.0 instead.
    assert int(O.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0x3F81
    assert int(O.f64_to_bf16(1.0 + 2.0 ** -8)) == 0x3F80
    assert int(O.f64_to_bf16(-0.0)) == 0x8000
    assert int(O.f64_to_bf16(1e39)) == 0x7F80


def test_e8m0_decode_vs_torch():
    b = np.arange(255, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(O.e8m0_decode(b), ref)
