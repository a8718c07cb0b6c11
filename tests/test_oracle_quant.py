"""Pins of the oracle's quantizer and bit packing, independent of its code.

The quantizer follows the stated op order (fp32 amax, fp16 scale, rint of the
fp32 quotient, clamp).  Each pin below would catch a plausible slip: a wrong
qmax, truncation instead of rounding, a dropped clamp, a swapped nibble, a
negative shift in the 3-bit codec (trefon.com "Matematyka cache KV", section
"Dlaczego cache trudniej skwantyzowac niz wagi": the 3-bit codec bug).
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import kvq_oracle as O


def round_to_binary(fr: Fraction, mant_bits: int, emin: int, emax: int) -> Fraction:
    """Exact IEEE round-to-nearest-even of a rational to a binary format with
    `mant_bits` fraction bits, minimum normal exponent emin, max exponent emax
    (overflow returns None).  Written from the IEEE 754 definition."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - mant_bits)
    q, r = divmod(a, ulp)
    q = int(q)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    v = q * ulp
    if v >= Fraction(2) ** (emax + 1):
        return None
    return sign * v


def to_f32(fr):
    return round_to_binary(fr, 23, -126, 127)


def to_f16(fr):
    return round_to_binary(fr, 10, -14, 15)


@pytest.mark.parametrize("val,expect", [
    (Fraction(1) + Fraction(1, 2 ** 11), Fraction(1)),                       # tie -> even (down)
    (Fraction(1) + Fraction(3, 2 ** 11), Fraction(1) + Fraction(1, 2 ** 9)),  # tie -> even (up)
    (Fraction(65519), Fraction(65504)),
    (Fraction(1, 2 ** 25), Fraction(0)),                                      # half the smallest subnormal -> 0
    (Fraction(3, 2 ** 26), Fraction(1, 2 ** 24)),
])
def test_fp16_rounding_matches_ieee_definition(val, expect):
    assert to_f16(val) == expect
    got = np.float32(float(val)).astype(np.float16)
    assert Fraction(float(got)) == expect


def test_fp16_rounding_random_against_definition():
    rng = np.random.default_rng(1)
    xs = (rng.standard_normal(4000) * 10.0 ** rng.integers(-7, 4, 4000)).astype(np.float32)
    got = xs.astype(np.float16)
    for x, g in zip(xs, got):
        assert Fraction(float(g)) == to_f16(Fraction(float(x))), x


@pytest.mark.parametrize("bits", [8, 4, 3, 2])
def test_scale_follows_two_step_rounding(bits):
    rng = np.random.default_rng(bits)
    x = (rng.standard_normal((300, 32)) * rng.uniform(1e-3, 50, (300, 1))).astype(np.float32)
    s16, _ = O.quantize(x, bits)
    for row, s in zip(x, s16):
        amax = max(abs(Fraction(float(v))) for v in row)
        s32 = to_f32(amax / O.QMAX[bits])
        expect = to_f16(min(s32, Fraction(65504)))
        assert Fraction(float(s)) == expect


@pytest.mark.parametrize("bits", [8, 4, 3, 2])
def test_codes_are_nearest_grid_point(bits):
    """Brute force: each code minimizes |x - c*s| over every allowed code,
    ties to the even code."""
    qmax = O.QMAX[bits]
    rng = np.random.default_rng(10 + bits)
    x = (rng.standard_normal((40, 32)) * 3).astype(np.float32)
    # plant exact half-way points to exercise ties
    s16, _ = O.quantize(x, bits)
    for i in range(0, 40, 4):
        s = float(s16[i])
        x[i, 1] = np.float32(0.5 * s)
        x[i, 2] = np.float32(-1.5 * s) if qmax >= 2 else np.float32(-0.5 * s)
    s16, codes = O.quantize(x, bits)
    for row, s, crow in zip(x, s16, codes):
        S = Fraction(float(s))
        for v, c in zip(row, crow):
            V = Fraction(float(v))
            errs = {k: abs(V - k * S) for k in range(-qmax, qmax + 1)}
            best = min(errs.values())
            assert errs[int(c)] == best, (v, c)
            ties = [k for k, e in errs.items() if e == best]
            if len(ties) > 1:
                assert int(c) % 2 == 0


@pytest.mark.parametrize("bits", [8, 4, 3, 2])
def test_error_bound_half_scale(bits):
    """|x - code*scale| <= scale/2, plus the clamp margin amax - qmax*scale
    (the fp16 scale may round below amax/qmax by up to 2^-11 relative)."""
    qmax = O.QMAX[bits]
    rng = np.random.default_rng(20 + bits)
    x = (rng.standard_normal((2000, 32)) * rng.lognormal(0, 2, (2000, 1))).astype(np.float32)
    s16, codes = O.quantize(x, bits)
    xh = O.dequantize_f64(s16, codes)
    s = s16.astype(np.float64)[:, None]
    amax = np.abs(x).max(-1, keepdims=True).astype(np.float64)
    margin = np.maximum(0.0, amax - qmax * s)
    err = np.abs(x - xh)
    assert np.all(err <= s / 2 * (1 + 2 ** -20) + margin)
    assert np.all(margin <= qmax * s * 2 ** -11 * (1 + 1e-9))


@pytest.mark.parametrize("bits", [8, 4, 3, 2])
def test_representable_grid_round_trips_exactly(bits):
    qmax = O.QMAX[bits]
    rng = np.random.default_rng(30 + bits)
    for e in (-12, -3, 0, 5, 10):
        s = 2.0 ** e
        c = rng.integers(-qmax, qmax + 1, (50, 32))
        c[:, 0] = qmax * np.where(rng.random(50) < 0.5, 1, -1)
        x = (c * s).astype(np.float32)
        s16, codes = O.quantize(x, bits)
        assert np.all(s16.astype(np.float64) == s)
        assert np.array_equal(codes.astype(np.int64), c)
    # through fp16 and bf16 inputs too (the grid is exact in both)
    x16 = (c * 0.25).astype(np.float16)
    s16, codes = O.quantize(O.f16_bits_to_f32(x16.view(np.uint16)), bits)
    assert np.array_equal(codes.astype(np.int64), c)


def test_zero_and_tiny_blocks_give_zero_codes():
    x = np.zeros((2, 32), np.float32)
    x[1, 3] = np.float32(2.0 ** -30)  # amax/7 rounds to a zero fp16 scale
    s16, codes = O.quantize(x, 4)
    assert np.all(s16 == 0) and np.all(codes == 0)


def test_scale_saturates_at_fp16_max():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.float32(1e6)
    x[0, 1] = np.float32(-3e5)
    x[0, 2] = np.float32(1000.0)
    s16, codes = O.quantize(x, 4)
    assert float(s16[0]) == 65504.0
    assert codes[0, 0] == 7 and codes[0, 1] == -5 and codes[0, 2] == 0


def _expected_int(codes, bits):
    """The packed block as one little-endian integer, built bit by bit."""
    total = 0
    for j, c in enumerate(codes):
        u = (int(c) & 0xFF) if bits == 8 else int(c) + (1 << (bits - 1))
        total |= u << (bits * j)
    return total


@pytest.mark.parametrize("bits,G", [(8, 32), (4, 32), (4, 128), (3, 128), (2, 32)])
def test_pack_every_code_at_every_position(bits, G):
    qmax = O.QMAX[bits]
    base = np.full(G, -qmax + 1 if qmax > 1 else 0, np.int64)
    per_word = {8: 1, 4: 2, 3: 8, 2: 4}[bits]
    for j in range(min(G, 2 * per_word)):
        for c in range(-qmax, qmax + 1):
            codes = base.copy()
            codes[j] = c
            packed = O.pack(codes[None], bits)[0]
            assert len(packed) == G * bits // 8
            assert int.from_bytes(bytes(packed), "little") == _expected_int(codes, bits)
            assert np.array_equal(O.unpack(packed[None], bits, G)[0].astype(np.int64), codes)


def test_three_bit_positions_three_to_seven_survive():
    """The codec bug described on trefon.com corrupted values 3-7 of each
    8-group (bit offsets >= 8, reached with a negative shift).  Values there
    must land at bits 9..23 of the 24-bit word and round-trip."""
    for c in range(-3, 4):
        codes = np.zeros(128, np.int64)
        codes[3::8] = c
        codes[7::8] = -c
        codes[5::8] = 3
        packed = O.pack(codes[None], 3)[0]
        w = int.from_bytes(bytes(packed[:3]), "little")
        assert (w >> 9) & 7 == c + 4
        assert (w >> 21) & 7 == -c + 4
        assert (w >> 15) & 7 == 7
        assert np.array_equal(O.unpack(packed[None], 3, 128)[0].astype(np.int64), codes)


@pytest.mark.parametrize("bits,G", [(8, 32), (4, 32), (4, 128), (3, 128), (2, 32)])
def test_block_is_scale_then_codes(bits, G):
    rng = np.random.default_rng(bits * G)
    x = rng.standard_normal((5, G)).astype(np.float32)
    blob = O.encode_blocks(x, bits)
    assert blob.shape == (5, O.block_bytes(bits, G))
    s16, codes = O.quantize(x, bits)
    for i in range(5):
        sbits = int.from_bytes(bytes(blob[i, :2]), "little")
        assert sbits == int(np.asarray(s16[i], np.float16).view(np.uint16))
    s2, c2 = O.decode_blocks(blob, bits, G)
    assert np.array_equal(s2.view(np.uint16), s16.view(np.uint16))
    assert np.array_equal(c2, codes)
