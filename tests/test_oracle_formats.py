"""Pins for the oracle's scalar format conversions (CPU only).

Every expectation here comes from somewhere other than the oracle's own code:
hand derivations written out beside the value, tables decoded from the bit
layout of each format by this file's own decoder, nearest-value search over
those tables, closed forms on the bit patterns, and torch's float8_e4m3fn
conversion as a third opinion.
"""
import math

import numpy as np
import pytest
import torch

import oracle

# --------------------------------------------------------------------------
# Independent decoders (bit layout -> value), written from the format
# definitions, not from the oracle.
# --------------------------------------------------------------------------


def e4m3_table():
    c = np.arange(256)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (c & 7 == 7), np.nan, mag)
    return sign * mag


def e2m1_table():
    c = np.arange(16)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def nearest_even(v, pos_values, sign_bit):
    """Code of the nearest value in pos_values (ascending, code i = value i),
    ties to the even code, saturating at the largest, sign bit OR-ed in for
    negative inputs (including -0)."""
    a = np.abs(v)
    n = len(pos_values)
    idx = np.clip(np.searchsorted(pos_values, a), 1, n - 1)
    lo, hi = pos_values[idx - 1], pos_values[idx]
    dlo, dhi = a - lo, hi - a
    code = np.where(dlo < dhi, idx - 1,
                    np.where(dhi < dlo, idx, np.where((idx - 1) % 2 == 0, idx - 1, idx)))
    code = np.where(a >= pos_values[-1], n - 1, code)
    code = np.where(a == 0, 0, code)
    return (code | np.where(np.signbit(v), sign_bit, 0)).astype(np.uint8)


E4M3 = e4m3_table()
E4M3_POS = E4M3[:0x7F]          # codes 0x00..0x7E, ascending
E2M1 = e2m1_table()
E2M1_POS = E2M1[:8]


def test_e4m3_table_pins():
    # Hand values from the E4M3 bit layout (bias 7, 3 mantissa bits).
    assert E4M3[0x7E] == 448.0          # 0 1111 110 = 1.75 * 2^8
    assert E4M3[0x08] == 2.0 ** -6      # smallest normal
    assert E4M3[0x01] == 2.0 ** -9      # smallest subnormal
    assert E4M3[0x38] == 1.0            # 0 0111 000
    assert E4M3[0x30] == 0.5
    assert E4M3[0xFE] == -448.0
    assert np.isnan(E4M3[0x7F]) and np.isnan(E4M3[0xFF])
    assert np.all(np.diff(E4M3_POS) > 0)
    # Third opinion: torch's own float8_e4m3fn decode.
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(t), np.isnan(E4M3))
    ok = ~np.isnan(E4M3)
    np.testing.assert_array_equal(t[ok], E4M3[ok])


def test_e4m3_decode_matches_table():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if np.isnan(E4M3[c]):
            assert math.isnan(v)
        else:
            assert v == E4M3[c], hex(c)


def test_e4m3_hand_values():
    # x * 2^-e for the worked blocks: (value, expected code, derivation)
    cases = [
        (384.0, 0x7C, "1.5*2^8: exponent field 15, mantissa 4"),
        (12.8125, 0x55, "1.6015625*2^3, 4.8125 mantissa steps -> 5: 1.625*8 = 13"),
        (17.0, 0x58, "1.0625*2^4, 0.5 step: tie -> even mantissa 0 -> 16"),
        (19.0, 0x5A, "1.1875*2^4, 1.5 steps: tie -> even mantissa 2 -> 20"),
        (-38.5, 0xE2, "1.203125*2^5, 1.625 steps -> 2 -> -40"),
        (510.0, 0x7E, "above 448: saturates"),
        (448.0, 0x7E, "largest finite"),
        (2.0 ** -8, 0x02, "2 subnormal steps of 2^-9"),
        (3 * 2.0 ** -10, 0x02, "1.5 subnormal steps: tie -> even 2"),
        (2.0 ** -10, 0x00, "0.5 subnormal steps: tie -> even 0"),
        (-(2.0 ** -10), 0x80, "negative tie to zero keeps the sign"),
        (0.5, 0x30, "exponent field 6"),
        (-0.1875, 0xA4, "-1.5*2^-3: exponent field 4, mantissa 4"),
        (2.0 ** -6, 0x08, "smallest normal"),
        (-0.0, 0x80, "negative zero"),
        (0.0, 0x00, "zero"),
        (1e30, 0x7E, "far above range saturates"),
        (-1e30, 0xFE, "negative saturation"),
        (464.0, 0x7E, "half a step above 448 still saturates"),
    ]
    for v, code, why in cases:
        got = int(oracle.e4m3_encode([v])[0])
        assert got == code, f"{v}: got {got:#x} want {code:#x} ({why})"


@pytest.mark.parametrize("e_lo,e_hi", [(-127, -60), (-60, 0), (0, 60), (60, 120)])
def test_e4m3_encode_bruteforce(e_lo, e_hi):
    """Every finite bf16 pattern times 2^-e for every reachable scale
    exponent e, against nearest-value search over the decoded table."""
    bits = np.arange(65536, dtype=np.uint32)
    exp_field = (bits >> 7) & 0xFF
    bits = bits[exp_field != 0xFF]
    x = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    for e in range(e_lo, e_hi):
        v = np.ldexp(x, -e)
        want = nearest_even(v, E4M3_POS, 0x80)
        got = oracle.e4m3_encode(v)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"e={e}: v={v[bad[:4]]} got={got[bad[:4]]} want={want[bad[:4]]}"


def test_e4m3_encode_vs_torch():
    """torch's fp32 -> float8_e4m3fn cast (round to nearest even) of values
    already clamped to +-448 agrees with the oracle encoder."""
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(200000) * 50.0,
        rng.standard_normal(200000) * 2.0 ** -8,
        np.ldexp(rng.integers(-64, 64, 200000).astype(np.float64), rng.integers(-16, 6, 200000)),
    ]).astype(np.float32)
    clamped = np.clip(v, -448.0, 448.0)
    t = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v.astype(np.float64))
    np.testing.assert_array_equal(got, t)


def test_e2m1_table_and_hand_values():
    assert list(E2M1_POS) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        assert oracle.e2m1_decode(c) == E2M1[c]
    cases = [(6, 0x7), (3, 0x5), (-1.5, 0xB), (0.25, 0x0), (0.75, 0x2), (1.25, 0x2),
             (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5, 0x6), (7, 0x7), (-0.0, 0x8),
             (0.0, 0x0), (-100.0, 0xF), (0.2499, 0x0), (0.2501, 0x1)]
    for v, code in cases:
        assert int(oracle.e2m1_encode([v])[0]) == code, v


def test_e2m1_encode_bruteforce():
    grid = np.arange(-9 * 256, 9 * 256 + 1) / 256.0
    rng = np.random.default_rng(5)
    v = np.concatenate([grid, -grid, rng.standard_normal(100000) * 4, np.ldexp(1.0, np.arange(-150, 10))])
    np.testing.assert_array_equal(oracle.e2m1_encode(v), nearest_even(v, E2M1_POS, 0x8))


def test_e8m0_closed_form_all_bf16():
    """For a bf16 (or fp32) amax, floor(log2 amax) - 8 clamped at -127 and
    biased by 127 equals max(0, exponent field - 8): check the oracle's
    frexp-based rule against that bit-level closed form for every positive
    finite bf16 value, plus amax = 0."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    amax = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    want = np.maximum(0, ((bits >> 7) & 0xFF).astype(np.int64) - 8).astype(np.uint8)
    np.testing.assert_array_equal(oracle.e8m0_code(amax), want)
    assert oracle.e8m0_code([0.0])[0] == 0
    assert oracle.e8m0_code([3.0])[0] == 120           # floor(log2 3) = 1 -> 1-8+127
    assert oracle.e8m0_code([1.9921875 * 2.0 ** 127])[0] == 246   # largest finite bf16
    assert oracle.e8m0_code([2.0 ** -128])[0] == 0     # clamps at -127
    # Doubles outside the bf16 range still follow floor(log2) exactly.
    assert oracle.e8m0_code([2.0 ** 200])[0] == 254    # clamps at +127
    assert oracle.e8m0_code([2.0 ** 134 * 1.5])[0] == 253


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):   # NaN patterns widen to NaN
        want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    for b in list(range(0, 65536, 97)) + [0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F]:
        got = oracle.bf16_decode(b)
        if np.isnan(want[b]):
            assert math.isnan(got)
        else:
            assert got == want[b], hex(b)


def test_e8m0_rceil_is_the_smallest_non_saturating_scale():
    """Ceil rule over every positive finite bf16 amax: 2^e is the smallest
    power of two with amax / 2^e <= 448 (clamped at e = -127), and it equals
    the integer form max(0, E - 8 + [mantissa > 1.75]) on the bf16 fields."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32)               # positive, finite
    amax = (bits << 16).view(np.float32).astype(np.float64)
    codes = oracle.e8m0_code_rceil(amax).astype(np.int64)
    e = codes - 127
    assert np.all(amax / np.exp2(e.astype(np.float64)) <= 448.0)
    above = e > -127
    assert np.all(amax[above] / np.exp2(e[above] - 1.0) > 448.0)
    E = (bits >> 7).astype(np.int64)
    mant = (bits & 0x7F).astype(np.int64)
    assert np.array_equal(codes, np.maximum(0, E - 8 + (mant > 0x60)))
    assert oracle.e8m0_code_rceil([0.0])[0] == 0
    assert oracle.e8m0_code_rceil([448.0])[0] == 127 and oracle.e8m0_code_rceil([449.0])[0] == 128
