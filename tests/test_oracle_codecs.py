"""Pins for the oracle's element codecs (float8_e4m3fn and the E8M0 block scale).

Each check ties the oracle to something other than itself: the format's value
table, an exhaustive nearest-code search, or the defining inequality of the
block-scale rule.
"""
import math

import numpy as np
import pytest

import oracle as O
from workloads import bf16_bits_to_f32


def _all_magnitudes():
    """Value of every non-negative, non-NaN e4m3fn code, built from the
    format's fields (bias 7, 3 mantissa bits, E=0 subnormal)."""
    vals = []
    for code in range(0x7F):
        E, m = code >> 3, code & 7
        vals.append(m / 8 * 2.0 ** -6 if E == 0 else (1 + m / 8) * 2.0 ** (E - 7))
    return np.array(vals)


def test_decode_table_spot_values():
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
            0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x7C: 384.0, 0x7E: 448.0, 0xB8: -1.0,
            0xFE: -448.0}
    got = O.e4m3_decode(np.array(list(want), np.uint8))
    assert got.tolist() == list(want.values())
    assert math.copysign(1.0, O.e4m3_decode(np.array([0x80], np.uint8))[0]) == -1.0


def test_decode_nan_codes_and_monotonic():
    allv = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(allv).sum() == 2 and np.isnan(allv[0x7F]) and np.isnan(allv[0xFF])
    pos = allv[:0x7F]
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(pos, _all_magnitudes())
    np.testing.assert_array_equal(allv[0x80:0xFF], -pos)


def _nearest_code(v: np.ndarray) -> np.ndarray:
    """Brute force: nearest of the 127 magnitudes, ties to even mantissa,
    saturating to 448, sign copied."""
    mags = _all_magnitudes()
    a = np.abs(v)
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    tie = d == best
    cand = np.where(tie, np.arange(127)[None, :], 1000)
    even = np.where(tie & (np.arange(127)[None, :] % 2 == 0), np.arange(127)[None, :], 1000)
    code = np.where(even.min(axis=1) < 1000, even.min(axis=1), cand.min(axis=1))
    code = np.where(a >= 448.0, 0x7E, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_encode_matches_exhaustive_nearest_search_on_all_bf16():
    """Every finite bf16 value of magnitude 2^-13 .. 2^10 (every significand
    in every e4m3 binade, the subnormal range and the saturation range), both
    signs: the inputs the MX path hands to the encoder are such values."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = bf16_bits_to_f32(bits).astype(np.float64)
    keep = np.isfinite(vals) & (((np.abs(vals) >= 2.0 ** -13) & (np.abs(vals) < 2.0 ** 10))
                                | (vals == 0))
    v = vals[keep]
    assert v.size > 5000
    np.testing.assert_array_equal(O.e4m3_encode(v), _nearest_code(v))


def test_encode_midpoints_and_random():
    mags = _all_magnitudes()
    mids = (mags[1:] + mags[:-1]) / 2
    rng = np.random.default_rng(7)
    rnd = rng.standard_normal(20000) * np.exp2(rng.integers(-14, 10, 20000))
    v = np.concatenate([mids, -mids, mags, -mags, rnd, [448.0, 449.0, 463.9, 464.0, 480.0, 1e9,
                                                         -1e9, 2.0 ** -10, -(2.0 ** -10)]])
    np.testing.assert_array_equal(O.e4m3_encode(v), _nearest_code(v))


def test_encode_decode_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


def test_encode_nan():
    assert O.e4m3_encode(np.array([np.nan]))[0] in (0x7F, 0xFF)


@pytest.mark.parametrize("amax,e", [(1.0, -8), (448.0, 0), (511.0, 0), (512.0, 1), (256.0, 0),
                                    (255.0, -1), (3.0, -7), (0.0, -127),
                                    (2.0 ** -126, -127), (2.0 ** -119, -127),
                                    (2.0 ** -118, -126), (3.3895313892515355e38, 119)])
def test_mx_scale_exponent_values(amax, e):
    assert O.mx_scale_exponent(amax) == e


def test_mx_scale_exponent_defining_inequality_over_bf16():
    """For every positive finite bf16 amax, unless clamped at -127:
    2^(e+8) <= amax < 2^(e+9), i.e. amax * 2^-e lies in [256, 512)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    vals = bf16_bits_to_f32(bits).astype(np.float64)
    for a in vals[::37]:
        e = O.mx_scale_exponent(a)
        if e == -127:
            assert a < 2.0 ** -118
        else:
            assert 256.0 <= a * 2.0 ** -e < 512.0
