"""Pins of the oracle's OCP E4M3 codec: the format's defining values, exhaustive round trips,
ties and saturation, and torch's own float8_e4m3fn conversions (a library routine that shares no
code with the oracle)."""

import numpy as np
import torch

from oracle import e4m3_decode, e4m3_encode_f32


def test_defining_values():
    d = e4m3_decode
    assert d(0x7E) == 448.0                      # largest finite: S.1111.110
    assert d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6                  # smallest normal
    assert d(0x07) == 0.875 * 2.0 ** -6          # largest subnormal
    assert d(0x01) == 2.0 ** -9                  # smallest subnormal
    assert d(0x38) == 1.0                        # e = 7 (bias), m = 0
    assert d(0x39) == 1.125
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))
    vals = e4m3_decode(np.arange(256))
    assert np.isnan(vals).sum() == 2             # no infinities, two NaNs


def test_decode_matches_torch_float8_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3_decode(codes)
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.signbit(ours[~both_nan]), np.signbit(ref[~both_nan]))


def test_encode_decode_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(e4m3_encode_f32(vals), codes)


def test_ties_round_to_even_mantissa():
    enc = e4m3_encode_f32
    assert enc(np.float32(1.0625)) == 0x38       # halfway 1.0 (m=0) / 1.125 (m=1) -> even
    assert enc(np.float32(1.1875)) == 0x3A       # halfway 1.125 (m=1) / 1.25 (m=2) -> even
    assert enc(np.nextafter(np.float32(1.0625), np.float32(2))) == 0x39
    assert enc(np.nextafter(np.float32(1.1875), np.float32(0))) == 0x39
    # subnormal / normal boundary: halfway between 0x07 and 0x08 goes to 0x08 (even)
    mid = np.float32((0.875 * 2.0 ** -6 + 2.0 ** -6) / 2)
    assert enc(mid) == 0x08
    # half the smallest subnormal rounds to (signed) zero; just above it to 0x01
    assert enc(np.float32(2.0 ** -10)) == 0x00
    assert enc(np.float32(-(2.0 ** -10))) == 0x80
    assert enc(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01


def test_saturation_and_nan():
    enc = e4m3_encode_f32
    for x in (448.0, 449.0, 464.0, 479.0, 480.0, 1e30, np.inf):
        assert enc(np.float32(x)) == 0x7E
        assert enc(np.float32(-x)) == 0xFE
    assert enc(np.float32(np.nan)) == 0x7F


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 40,
        rng.standard_normal(50000).astype(np.float32) * 1e-2,
        (rng.uniform(-448, 448, 50000)).astype(np.float32),
        e4m3_decode(np.arange(0, 0x7F)).astype(np.float32),
    ])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode_f32(x), ref)
