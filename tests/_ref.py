"""Independent reference arithmetic used by the oracle's pin tests.

Everything here is exact rational arithmetic (fractions.Fraction) or mpmath at high
precision, written separately from oracle.cpp, so that a mistake in the oracle's
double-precision code (a dropped term, a wrong sign, a transposed operand, a wrong
rounding rule) shows up as a mismatch.
"""
from __future__ import annotations

from fractions import Fraction

import mpmath
import numpy as np

mpmath.mp.dps = 50


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit-twiddle round-to-nearest-even of fp32 -> bf16 (non-NaN inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_float(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def frac(x) -> Fraction:
    """Exact Fraction of a float or an mpmath mpf."""
    if isinstance(x, mpmath.mpf):
        sign, man, exp, _ = x._mpf_
        if not man and exp == 0 and sign == 0:
            return Fraction(0)
        v = Fraction(int(man)) * (Fraction(2) ** int(exp))
        return -v if sign else v
    return Fraction(float(x))


def _round_bits(x: Fraction, sig_bits: int, min_q: int, max_exp: int) -> Fraction | float:
    """Nearest number with `sig_bits` significant bits (spacing >= 2^min_q), ties to even.
    Returns a Fraction, or +-inf on overflow (|r| >= 2^max_exp)."""
    if x == 0:
        return Fraction(0)
    ax = abs(x)
    # e with 2^(e-1) <= ax < 2^e
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    while Fraction(2) ** e <= ax:
        e += 1
    while Fraction(2) ** (e - 1) > ax:
        e -= 1
    q = max(e - sig_bits, min_q)
    scaled = ax / (Fraction(2) ** q)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * Fraction(2) ** q
    if r >= Fraction(2) ** max_exp:
        return float("inf") if x > 0 else float("-inf")
    return r if x > 0 else -r


def rnd_bf16(x) -> float:
    """Exact value -> nearest bf16 (as a float)."""
    r = _round_bits(frac(x) if not isinstance(x, Fraction) else x, 8, -133, 128)
    return float(r)


def rnd_f32(x) -> float:
    r = _round_bits(frac(x) if not isinstance(x, Fraction) else x, 24, -149, 128)
    return float(r)


def bf16_bits(v: float) -> int:
    """Bit pattern of a float that is exactly a bf16 number."""
    b = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
    assert float(bf16_to_float(np.uint16(b))) == v or np.isnan(v)
    return b


def near_tie_bf16(x, rel: float = 1e-12) -> bool:
    """True when exact value x lies within rel of a bf16 rounding midpoint."""
    x = frac(x) if not isinstance(x, Fraction) else x
    if x == 0:
        return False
    lo = rnd_bf16(x)
    # midpoints around x: neighbours of lo at half spacing
    ax = abs(float(x))
    e = np.frexp(ax)[1]
    q = 2.0 ** max(e - 8, -133)
    for m in (abs(lo) - q / 2, abs(lo) + q / 2):
        if abs(ax - m) <= rel * ax:
            return True
    return False
