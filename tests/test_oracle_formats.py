"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle's own decoder/encoder against something other
than itself: numpy's binary16, torch's float8_e4m3fn, the printed value
tables under tests/golden/, or closed-form properties of round-to-nearest-even.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_f16_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(codes)
    ref = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # signed zero survives
    assert np.signbit(ours[0x8000]) and ours[0x8000] == 0.0


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_to_f64(codes.numpy())
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_e4m3_landmarks_golden():
    for code_hex, val in _read_table("e4m3_landmarks.txt"):
        got = oracle.e4m3_to_f64(np.array([int(code_hex, 16)], dtype=np.uint8))[0]
        assert got == float(val), (code_hex, got, val)


def test_e2m1_value_set_golden():
    for code, val in _read_table("e2m1_values.txt"):
        got = oracle.e2m1_to_f64(np.array([int(code)], dtype=np.uint8))[0]
        assert got == float(val), (code, got, val)


def test_e4m3_encode_round_trips_every_finite_code():
    vals = oracle.e4m3_table()
    for code in range(256):
        if np.isnan(vals[code]):
            continue
        enc = int(oracle.f64_to_e4m3(np.array([vals[code]]))[0])
        assert enc == code, (hex(code), vals[code], hex(enc))


def test_e4m3_encode_ties_go_to_even_code():
    vals = oracle.e4m3_table()
    pos = [c for c in range(0x00, 0x7F)]  # 0 .. 448 ascending
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (vals[lo] + vals[hi]) / 2.0
        enc = int(oracle.f64_to_e4m3(np.array([mid]))[0])
        assert enc == (lo if lo % 2 == 0 else hi), (hex(lo), hex(hi), mid, hex(enc))
        # just either side of the midpoint rounds to the nearer code
        eps = (vals[hi] - vals[lo]) * 1e-6
        assert int(oracle.f64_to_e4m3(np.array([mid - eps]))[0]) == lo
        assert int(oracle.f64_to_e4m3(np.array([mid + eps]))[0]) == hi


def test_e4m3_encode_saturates_and_matches_torch_in_range():
    big = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e6, -1e6, -460.0])
    enc = oracle.f64_to_e4m3(big)
    assert [int(e) for e in enc] == [0x7E] * 6 + [0xFE] * 2
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)])
    x = x[np.abs(x) < 440.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = oracle.f64_to_e4m3(x)
    assert np.array_equal(ours, ref)


def test_nvfp4_product_rounding_matches_torch_cast():
    """e4m3_rne_sat(e2m1(code) * e4m3(sf)) for every nibble and scale code,
    against torch's own float32 -> float8_e4m3fn cast (the float32 product is
    exact: at most 2 x 4 significant bits)."""
    nib = np.arange(16, dtype=np.uint8)
    sf = np.arange(256, dtype=np.uint8)
    e2 = oracle.e2m1_to_f64(nib)
    e4 = oracle.e4m3_table()
    prod = (e2[:, None] * e4[None, :])
    finite = ~np.isnan(prod)
    ours = oracle.f64_to_e4m3(np.where(finite, prod, 0.0))
    p32 = torch.from_numpy(np.where(finite, prod, 0.0)).to(torch.float32)
    in_range = (p32.abs() < 464.0).numpy()
    ref = p32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    m = finite & in_range
    assert np.array_equal(ours[m], ref[m])
    # products above the E4M3 range saturate to +-448
    sat = finite & ~in_range
    assert sat.any()
    assert set(int(v) for v in np.unique(ours[sat])) <= {0x7E, 0xFE}
