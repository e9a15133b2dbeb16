"""Pins for the oracle's E4M3 encode/decode (CPU only).

Independent anchors: the OCP OFP8 spec's named values (golden fixture),
torch's float8_e4m3fn conversions (a library routine), and brute-force
properties of round-to-nearest-even on the full code table.
"""

import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp_values.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def test_decode_spec_values():
    for code, val in _golden():
        got = e4m3.decode(np.array([code], dtype=np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_encode_spec_values():
    for code, val in _golden():
        if np.isnan(val):
            continue
        assert e4m3.encode(np.array([val]))[0] == code, hex(code)


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3.decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    assert np.array_equal(e4m3.encode(e4m3.decode(codes)), codes)


def test_exactly_two_nan_codes():
    nan = np.isnan(e4m3.decode(np.arange(256, dtype=np.uint8)))
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]


def test_midpoints_tie_to_even_and_interiors_to_nearest():
    pos = np.arange(0x00, 0x7F, dtype=np.uint8)          # 0 .. 448
    vals = e4m3.decode(pos)
    for c in range(len(pos) - 1):
        lo, hi = vals[c], vals[c + 1]
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        got = e4m3.encode(np.array([mid, -mid]))
        assert got[0] == even and got[1] == (even | 0x80), (c, mid)
        # strictly inside each half goes to that side
        qlo = lo + (hi - lo) * 0.25
        qhi = lo + (hi - lo) * 0.75
        got = e4m3.encode(np.array([qlo, qhi]))
        assert got[0] == c and got[1] == c + 1


def test_saturation_and_specials():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e6, np.inf, -np.inf, -1e30, np.nan, -np.nan])
    got = e4m3.encode(x)
    assert list(got[:6]) == [0x7E] * 6
    assert list(got[6:8]) == [0xFE, 0xFE]
    assert got[8] == 0x7F and got[9] == 0xFF


def test_underflow_keeps_sign_and_ties_even():
    t = 2.0 ** -10              # half the smallest subnormal: ties to 0 (even)
    got = e4m3.encode(np.array([t, -t, t * 1.0001, -1e-30, 0.0, -0.0]))
    assert list(got) == [0x00, 0x80, 0x01, 0x80, 0x00, 0x80]


def test_encode_matches_torch_random_float32():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 50,
        rng.standard_normal(50000).astype(np.float32) * 0.01,   # subnormal range
        rng.uniform(-448, 448, 50000).astype(np.float32),
    ])
    ours = e4m3.encode(x)
    clamped = torch.from_numpy(np.clip(x, -448, 448))
    ref = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_monotonic_dense_sweep():
    x = np.linspace(-500, 500, 400001)
    v = e4m3.decode(e4m3.encode(x))
    assert np.all(np.diff(v) >= 0)
    assert np.all(np.abs(v) <= 448)


def test_round_significand_matches_e4m3_normal_range():
    rng = np.random.default_rng(2)
    x = np.exp(rng.uniform(np.log(2.0 ** -6), np.log(440.0), 100000))
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(e4m3.round_significand(x, 4), ref)


def test_round_significand_scale_free():
    rng = np.random.default_rng(3)
    x = rng.uniform(0.01, 1.0, 10000)
    for k in (-20, -7, 5, 30):
        assert np.array_equal(e4m3.round_significand(x * 2.0 ** k, 4),
                              e4m3.round_significand(x, 4) * 2.0 ** k)
