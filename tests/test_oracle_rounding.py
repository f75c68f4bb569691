"""Pins for the oracle's single fp64 -> fp16 rounding (round to nearest, ties
to even, overflow to Inf, subnormals kept).

Checked by brute force against exact rational rounding written here from the
IEEE 754 binary16 definition, and against numpy's float64 -> float16 cast.
"""
from fractions import Fraction

import numpy as np

import oracle


def rne_fraction_to_f16_bits(x: Fraction) -> int:
    """Exact IEEE binary16 rounding of a rational (ties to even)."""
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a == 0:
        return sign
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (max(e, -14) - 10)      # spacing of binary16 near a
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * q
    if v >= 65536:
        return sign | 0x7C00
    if v < Fraction(2) ** -14:
        return sign | int(v / Fraction(2) ** -24)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    mant = int(v / Fraction(2) ** (e - 10)) - 1024
    return sign | ((e + 15) << 10) | mant


def all_finite_f16():
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16)
    keep = np.isfinite(v)
    return bits[keep], v[keep].astype(np.float64)


def test_every_fp16_value_is_a_fixed_point():
    bits, v = all_finite_f16()
    out = oracle.f64_to_f16(v).view(np.uint16)
    # -0 and +0 are both fixed points with their own sign
    assert np.array_equal(out, bits)


def test_midpoints_and_neighbours_brute_force():
    pos = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0                      # exact in fp64
    cases = np.concatenate([mid, np.nextafter(mid, -np.inf), np.nextafter(mid, np.inf)])
    cases = np.concatenate([cases, -cases])
    out = oracle.f64_to_f16(cases).view(np.uint16)
    # numpy's direct double -> half cast rounds to nearest even
    ref = cases.astype(np.float16).view(np.uint16)
    assert np.array_equal(out, ref)
    # and exact rational rounding on a deterministic subsample
    idx = np.linspace(0, cases.size - 1, 4000).astype(np.int64)
    for i in idx:
        assert int(out[i]) == rne_fraction_to_f16_bits(Fraction(float(cases[i]))), cases[i]


def test_overflow_and_underflow_edges():
    f = lambda x: int(oracle.f64_to_f16(np.array([x])).view(np.uint16)[0])
    assert f(65504.0) == 0x7BFF
    assert f(np.nextafter(65520.0, 0)) == 0x7BFF     # just below the midpoint
    assert f(65520.0) == 0x7C00                      # tie goes to even = Inf
    assert f(1e300) == 0x7C00 and f(-1e300) == 0xFC00
    assert f(np.inf) == 0x7C00
    assert f(2.0 ** -24) == 0x0001
    assert f(2.0 ** -25) == 0x0000                   # tie to even (zero)
    assert f(np.nextafter(2.0 ** -25, 1)) == 0x0001
    assert f(3 * 2.0 ** -25) == 0x0002               # 1.5 ulp: tie -> even (2)
    assert f(-0.0) == 0x8000
    assert (f(np.nan) & 0x7C00) == 0x7C00 and (f(np.nan) & 0x03FF) != 0


def test_random_doubles_against_numpy_and_fractions():
    rng = np.random.default_rng(1234)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 18, 200000))
    out = oracle.f64_to_f16(x).view(np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(out, ref)
    for i in range(0, 200000, 97):
        assert int(out[i]) == rne_fraction_to_f16_bits(Fraction(float(x[i])))
