"""Pins of the oracle's residual-stream step x_{i+1} = bf16(x_i + y_i) (CPU).

The step is an fp32 add of two bf16 values followed by rounding to bf16, nearest even.  It is
checked against values worked out by hand and against an independent exact computation:
Python fractions give the exact sum, which is rounded to fp32 and then to bf16 by
searching the neighbouring representable values (no bit tricks).
"""
from fractions import Fraction
import math

import numpy as np

from oracle import moe as omoe


def _bits(vals):
    return np.asarray(vals, dtype=np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)


def _val(bits):
    return float(omoe.bf16_to_f64(np.array([bits], np.uint16))[0])


def _round_to_grid(q: Fraction, mant_bits: int) -> Fraction:
    """Nearest value with `mant_bits` significant bits (normal range), ties to even."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - mant_bits + 1)
    n = a / ulp
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * ulp


def test_hand_worked_values():
    # 1.0 + 0.5 = 1.5 exactly
    assert _val(omoe.residual_next(_bits([1.0]), _bits([0.5]))[0]) == 1.5
    # 1 + 2^-8: exactly halfway between 1 and 1 + 2^-7 -> the even one, 1.0
    assert _val(omoe.residual_next(_bits([1.0]), _bits([2.0 ** -8]))[0]) == 1.0
    # 1 + 3 * 2^-8: halfway between 1 + 2^-7 and 1 + 2^-6 -> even mantissa, 1 + 2^-6
    r = omoe.residual_next(_bits([1.0 + 2.0 ** -7]), _bits([2.0 ** -8]))[0]
    assert _val(r) == 1.0 + 2.0 ** -6
    # x + (-x) = +0
    assert omoe.residual_next(_bits([3.25]), _bits([-3.25]))[0] == 0
    # rounding up into the next binade: (2 - 2^-7) + 2^-8 is halfway, odd last bit -> 2.0
    assert _val(omoe.residual_next(_bits([2.0 - 2.0 ** -7]), _bits([2.0 ** -8]))[0]) == 2.0


def test_matches_exact_double_rounding():
    rng = np.random.default_rng(5)
    # bf16 values over a few binades, including far-apart exponents (the fp32 add rounds)
    a = (rng.standard_normal(4000) * np.exp2(rng.integers(-12, 12, 4000))).astype(np.float32)
    b = (rng.standard_normal(4000) * np.exp2(rng.integers(-12, 12, 4000))).astype(np.float32)
    ab, bb = _bits(a), _bits(b)
    got = omoe.residual_next(ab, bb)
    for i in range(len(a)):
        exact = Fraction(_val(ab[i])) + Fraction(_val(bb[i]))
        want = _round_to_grid(_round_to_grid(exact, 24), 8)
        assert Fraction(_val(got[i])) == want, (i, _val(ab[i]), _val(bb[i]))
