"""Pins of the oracle's FP8 (E4M3) cache format (CPU only).

- The format's fixed points: largest finite 448 (0x7E), smallest normal 2^-6 (0x08),
  smallest subnormal 2^-9 (0x01), NaN 0x7F / 0xFF, and all 256 decoded values against
  PyTorch's float8_e4m3fn (a library cross-check of the same encoding).
- Encoding: round trip of every finite code, ties to the even code at every midpoint,
  saturation beyond 448, agreement with PyTorch's conversion for in-range values, and the
  vectorised encoder equal to the scalar definition.
- Quantised writes: the division happens in binary32 before the E4M3 rounding (a case
  where rounding the exact quotient instead gives another code), padding slots skipped.
"""
import math

import numpy as np
import torch

from oracle.fp8 import (DECODE_TABLE, MAX_E4M3, dequantize, e4m3_decode, e4m3_encode, e4m3_encode_array,
                        kv_write_fp8_ref, quantize)


def test_format_fixed_points():
    assert e4m3_decode(0x7E) == 448.0 == MAX_E4M3
    assert e4m3_decode(0xFE) == -448.0
    assert e4m3_decode(0x08) == 2.0 ** -6
    assert e4m3_decode(0x07) == 7 / 8 * 2.0 ** -6  # largest subnormal
    assert e4m3_decode(0x01) == 2.0 ** -9
    assert e4m3_decode(0x00) == 0.0 and math.copysign(1.0, e4m3_decode(0x80)) == -1.0
    assert math.isnan(e4m3_decode(0x7F)) and math.isnan(e4m3_decode(0xFF))
    assert e4m3_decode(0x38) == 1.0  # exponent field 7 = bias


def test_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    theirs = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(DECODE_TABLE)
    assert np.array_equal(nan, np.isnan(theirs)) and nan.sum() == 2
    assert np.array_equal(DECODE_TABLE[~nan], theirs[~nan])


def test_round_trip_ties_and_saturation():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert e4m3_encode(DECODE_TABLE[c]) == c
    for c in range(0x7E):  # midpoint between consecutive non-negative codes: the even one
        mid = (DECODE_TABLE[c] + DECODE_TABLE[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert e4m3_encode(mid) == want
        assert e4m3_encode(-mid) == want | 0x80
        assert e4m3_encode(np.nextafter(mid, 0)) == c and e4m3_encode(np.nextafter(mid, 1e9)) == c + 1
    for x in (448.0, 463.99, 464.0, 480.0, 1e6, np.float32(3.4e38)):
        assert e4m3_encode(x) == 0x7E and e4m3_encode(-x) == 0xFE


def test_vectorised_encoder_and_torch_agree():
    rng = np.random.default_rng(1)
    mids = (DECODE_TABLE[:0x7E] + DECODE_TABLE[1:0x7F]) / 2
    x = np.concatenate([rng.standard_normal(30000) * rng.choice([1e-4, 1e-2, 1, 30, 300, 3000], 30000),
                        mids, -mids, DECODE_TABLE[:0x7F], [0.0, -0.0, 500.0, -1e9]]).astype(np.float32)
    v = e4m3_encode_array(x)
    assert np.array_equal(v, np.array([e4m3_encode(t) for t in x], np.uint8))
    inr = np.abs(x) < 448
    t = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(t, v[inr])


def test_quantize_divides_in_binary32_first():
    """x = float32(m * s) for an E4M3 midpoint m: the exact quotient x / s sits just off the
    midpoint while the binary32 quotient lands on it, so the two roundings differ; the
    oracle must take the binary32 one (a tie, resolved to the even code)."""
    from fractions import Fraction

    m = (DECODE_TABLE[0x38] + DECODE_TABLE[0x39]) / 2  # 1.0625, between codes 0x38 (even) and 0x39
    rng = np.random.default_rng(7)
    found = 0
    for _ in range(2000):
        sc = np.float32(rng.uniform(0.003, 0.05))
        x = np.float32(m * float(sc))
        exact = Fraction(float(x)) / Fraction(float(sc))
        q32 = np.float32(x) / np.float32(sc)
        if float(q32) == m and exact != Fraction(m):
            want_exact = 0x39 if exact > Fraction(m) else 0x38
            assert e4m3_encode(float(q32)) == 0x38  # the tie goes to the even code
            got = quantize(np.array([x]), sc)[0]
            assert got == 0x38
            found += want_exact != got
    assert found >= 3  # cases where rounding the exact quotient would give the other code


def test_kv_write_fp8_ref_places_codes_and_skips_padding():
    B, H, D = 4, 2, 16
    kc = np.zeros((3, B, H, D), np.uint8)
    vc = np.zeros_like(kc)
    rng = np.random.default_rng(2)
    k = rng.standard_normal((3, H, D)).astype(np.float32)
    v = rng.standard_normal((3, H, D)).astype(np.float32)
    kv_write_fp8_ref(kc, vc, k, v, [5, -1, 11], B, 0.25, 0.5)
    assert np.array_equal(kc[1, 1], quantize(k[0], 0.25)) and np.array_equal(vc[2, 3], quantize(v[2], 0.5))
    assert np.count_nonzero(kc.reshape(12, -1).any(axis=1)) == 2
    back = dequantize(kc[1, 1], 0.25)
    assert np.max(np.abs(back - k[0])) <= 0.25 * 2.0 ** -4 * 448  # within half an ulp at the top binade
    assert np.all(np.abs(back - k[0]) <= np.maximum(np.abs(k[0]) * 2.0 ** -4, 0.25 * 2.0 ** -10))
