"""Pins for the oracle's number formats (CPU only).

The E4M3 encoder and decoder are checked against (a) values fixed by the
OCP FP8 E4M3FN bit layout, derived by hand below, and (b) PyTorch's own
float8_e4m3fn conversion routines, an implementation independent of the
oracle.  PyTorch's cast rounds to nearest-even but turns values that round
past 448 into NaN instead of saturating, so the library comparison covers the
non-saturating range |x| <= 464 and saturation is pinned separately.
"""
import math

import numpy as np
import pytest
import torch

import oracle

# (code, value): sign | exponent(4, bias 7) | mantissa(3); exponent 0 holds
# subnormals m * 2^-9.
HAND_CODES = [
    (0x00, 0.0),
    (0x01, 2.0 ** -9),               # e=0 m=1: smallest subnormal
    (0x07, 7 * 2.0 ** -9),           # e=0 m=7: largest subnormal
    (0x08, 2.0 ** -6),               # e=1 m=0: smallest normal
    (0x0F, 1.875 * 2.0 ** -6),       # e=1 m=7
    (0x30, 0.5),                     # e=6
    (0x38, 1.0),                     # e=7 m=0
    (0x39, 1.125),                   # e=7 m=1
    (0x3C, 1.5),                     # e=7 m=4
    (0x40, 2.0),                     # e=8
    (0x44, 3.0),                     # e=8 m=4
    (0x4C, 6.0),                     # e=9 m=4
    (0x70, 128.0),                   # e=14
    (0x77, 240.0),                   # e=14 m=7
    (0x78, 256.0),                   # e=15 m=0
    (0x7D, 416.0),                   # e=15 m=5
    (0x7E, 448.0),                   # e=15 m=6: largest finite
    (0xB8, -1.0),
    (0xFE, -448.0),
]


def test_decode_hand_codes():
    for code, val in HAND_CODES:
        assert oracle.e4m3_decode(np.array([code], np.uint8))[0] == val, hex(code)
    z = oracle.e4m3_decode(np.array([0x80], np.uint8))[0]
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    for nan_code in (0x7F, 0xFF):
        assert math.isnan(oracle.e4m3_decode(np.array([nan_code], np.uint8))[0])


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert nan.sum() == 2


def test_encode_round_trips_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_hand_midpoints_tie_to_even():
    cases = [
        (1.0625, 0x38),        # between 1.0 (m=0) and 1.125 (m=1) -> even m=0
        (1.1875, 0x3A),        # between 1.125 (m=1) and 1.25 (m=2) -> m=2
        (2.0 ** -10, 0x00),    # between 0 and 2^-9 -> 0
        (3 * 2.0 ** -10, 0x02),  # between 1 and 2 subnormal units -> 2
        (7.5 * 2.0 ** -9, 0x08),  # between largest subnormal and 2^-6 -> 0x08
        (432.0, 0x7E),         # between 416 (m=5) and 448 (m=6) -> 448
        (464.0, 0x7E),         # midpoint of 448 and the (absent) 480 -> 448
        (-1.0625, 0xB8),
    ]
    for v, code in cases:
        assert int(oracle.e4m3_encode(np.array([v], np.float32))[0]) == code, v
        up = np.nextafter(np.float32(abs(v)), np.float32(np.inf))
        dn = np.nextafter(np.float32(abs(v)), np.float32(0))
        sign = 0x80 if v < 0 else 0
        if abs(v) < 448.0:
            lo = int(oracle.e4m3_encode(np.array([dn], np.float32))[0]) & 0x7F
            hi = int(oracle.e4m3_encode(np.array([up], np.float32))[0]) & 0x7F
            assert hi - lo == 1, (v, lo, hi)
        del sign


def test_encode_saturates_and_keeps_nan_and_signed_zero():
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, 3.0e38, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    nan = np.array([np.nan, -np.nan], np.float32)
    assert np.all((oracle.e4m3_encode(nan) & 0x7F) == 0x7F)
    tiny = np.array([0.0, 1e-30, 2.0 ** -10, 1e-45], np.float32)
    assert np.all(oracle.e4m3_encode(tiny) == 0x00)
    assert np.all(oracle.e4m3_encode(-tiny) == 0x80)


def _torch_e4m3(vals: np.ndarray) -> np.ndarray:
    return torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_on_every_fp32_pattern_in_range():
    """Every FP32 bit pattern from 2^-11 up to 464 (both signs), plus a
    strided sample of the patterns below 2^-11, against torch's cast."""
    lo = int(np.array([2.0 ** -11], np.float32).view(np.uint32)[0])
    hi = int(np.array([464.0], np.float32).view(np.uint32)[0])
    chunk = 1 << 24
    start = lo
    while start <= hi:
        n = min(chunk, hi - start + 1)
        bits = np.arange(start, start + n, dtype=np.uint32)
        vals = bits.view(np.float32)
        ours = oracle.e4m3_encode_bits(start, n)
        assert np.array_equal(ours, _torch_e4m3(vals)), hex(start)
        neg_bits = bits | np.uint32(0x80000000)
        ours_n = oracle.e4m3_encode_bits(start | 0x80000000, n)
        assert np.array_equal(ours_n, _torch_e4m3(neg_bits.view(np.float32))), hex(start)
        start += n
    small = np.arange(0, lo, 4099, dtype=np.uint32)
    for b in (small, small | np.uint32(0x80000000)):
        assert np.array_equal(oracle.e4m3_encode(b.view(np.float32)), _torch_e4m3(b.view(np.float32)))


def test_bf16_round_trip_and_rounding():
    x = torch.randn(100000, generator=torch.Generator().manual_seed(5)) * 37.0
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.f32_to_bf16(float(v)) for v in x[:2000].numpy()], np.uint16)
    assert np.array_equal(ours, ref[:2000])
    back = oracle.bf16_to_f32(ref)
    assert np.array_equal(back, x.to(torch.bfloat16).to(torch.float32).numpy())
