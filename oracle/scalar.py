"""Second, scalar formulation of the MX and blockwise quantizers (pure Python).

TEST INFRASTRUCTURE ONLY (see the package docstring).

This module restates the same rules as ``oracle.mx`` / ``oracle.blockwise``
in a different way, so that a slip in one formulation shows up as a
disagreement with the other:

* the shared exponent is read off the BF16 bit pattern (exponent field, and
  the mantissa's leading bit for subnormals) instead of ``frexp``;
* element rounding is built the IEEE way -- find the binade, divide by its
  quantum, round half to even on an exact rational, re-encode the bits --
  instead of a nearest-neighbour search over the value table;
* fp32 operations of the blockwise rule are rounded from exact rationals
  (``fractions.Fraction``) rather than performed by NumPy.

Only meant for small inputs (hand-worked blocks, sweeps of single values).
"""

from __future__ import annotations

from fractions import Fraction
import math

# format parameters: (exponent bits, mantissa bits, bias, max finite code magnitude)
_FMT = {
    "e2m1": dict(mbits=1, bias=1, emin=0, max_val=Fraction(6), sign_bit=3),
    "e4m3": dict(mbits=3, bias=7, emin=-6, max_val=Fraction(448), sign_bit=7),
}


def bf16_value(bits: int) -> Fraction:
    s = (bits >> 15) & 1
    E = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if E == 0xFF:
        raise ValueError("non-finite input")
    if E == 0:
        v = Fraction(m, 1 << 7) * Fraction(1, 1 << 126)
    else:
        v = (1 + Fraction(m, 1 << 7)) * Fraction(2) ** (E - 127)
    return -v if s else v


def floor_log2_bf16_magnitude(bits: int):
    """floor(log2 |x|) straight from the BF16 fields; None for zero."""
    E = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if E:
        return E - 127
    if m == 0:
        return None
    return -133 + (m.bit_length() - 1)           # subnormal: m * 2^-133


def mx_scale_exponent(block_bits, elem: str, rule: str = "ocp") -> int:
    mags = [b & 0x7FFF for b in block_bits]
    amax_bits = max(mags)                          # magnitude order == integer order
    fl = floor_log2_bf16_magnitude(amax_bits)
    if fl is None:
        return -127
    if rule == "round_up":
        # walk powers of two: the smallest 2^e with maxval * 2^e >= amax
        amax = bf16_value(amax_bits)
        e = 0
        while _FMT[elem]["max_val"] * Fraction(2) ** e < amax:
            e += 1
        while _FMT[elem]["max_val"] * Fraction(2) ** (e - 1) >= amax:
            e -= 1
        return max(-127, min(127, e))
    emax = 2 if elem == "e2m1" else 8
    return max(-127, min(127, fl - emax))


def _round_half_even(q: Fraction) -> int:
    f = math.floor(q)
    r = q - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        return f + 1
    return f


def encode(v: Fraction, elem: str, negative: bool) -> int:
    """Round the exact value v to the element format (RNE, saturating) and
    return its code, with the sign bit taken from ``negative``."""
    p = _FMT[elem]
    a = abs(v)
    code_mag = 0
    if a != 0:
        # binade exponent: exact floor(log2(a)) for a rational, then not
        # below the smallest normal exponent
        e = a.numerator.bit_length() - a.denominator.bit_length()
        if Fraction(2) ** e > a:
            e -= 1
        e = max(e, p["emin"])
        quantum = Fraction(2) ** (e - p["mbits"])
        n = _round_half_even(a / quantum)          # integer multiple of quantum
        val = n * quantum
        if val > p["max_val"]:
            val = p["max_val"]
        if val == 0:
            code_mag = 0
        else:
            # re-encode val into (E, m)
            ev = val.numerator.bit_length() - val.denominator.bit_length()
            if Fraction(2) ** ev > val:
                ev -= 1
            if ev < p["emin"]:                      # subnormal
                m = val / (Fraction(2) ** (p["emin"] - p["mbits"]))
                Ef = 0
            else:
                m = (val / Fraction(2) ** ev - 1) * (1 << p["mbits"])
                Ef = ev + p["bias"]
            assert m.denominator == 1
            code_mag = (Ef << p["mbits"]) | int(m)
    return code_mag | ((1 << p["sign_bit"]) if negative else 0)


def quantize_block_mx(block_bits, elem: str, rule: str = "ocp"):
    """One 32-element BF16 block -> (scale byte, list of codes)."""
    e = mx_scale_exponent(block_bits, elem, rule)
    codes = []
    for b in block_bits:
        v = bf16_value(b) / (Fraction(2) ** e)
        codes.append(encode(v, elem, negative=bool((b >> 15) & 1)))
    return e + 127, codes


def round_to_f32(v: Fraction) -> Fraction:
    """Correctly rounded (RNE) fp32 value of an exact rational (normal and
    subnormal range; no overflow handling needed here)."""
    if v == 0:
        return Fraction(0)
    neg = v < 0
    a = -v if neg else v
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    r = _round_half_even(a / quantum) * quantum
    return -r if neg else r


F32_1EM4 = round_to_f32(Fraction(1, 10000))


def quantize_block_bw(block_bits, pow2: bool = False):
    """One blockwise-FP8 block (any number of BF16 values sharing one scale)
    -> (fp32 scale as a Fraction, list of E4M3 codes).  pow2: the scale is
    the smallest power of two s with 448 * s >= a, found by walking exact
    powers of two."""
    vals = [bf16_value(b) for b in block_bits]
    amax = max(abs(v) for v in vals)
    a = max(amax, F32_1EM4)
    if pow2:
        s = Fraction(1)
        while 448 * s < a:
            s *= 2
        while 448 * (s / 2) >= a:
            s /= 2
    else:
        s = round_to_f32(a / 448)
    codes = []
    for b, v in zip(block_bits, vals):
        q = round_to_f32(v / s)
        codes.append(encode(q, "e4m3", negative=bool((b >> 15) & 1)))
    return s, codes


def decode_code(code: int, elem: str) -> Fraction:
    p = _FMT[elem]
    sign = (code >> p["sign_bit"]) & 1
    mag = code & ((1 << p["sign_bit"]) - 1)
    Ef = mag >> p["mbits"]
    m = mag & ((1 << p["mbits"]) - 1)
    if Ef == 0:
        v = m * Fraction(2) ** (p["emin"] - p["mbits"])
    else:
        v = (1 + Fraction(m, 1 << p["mbits"])) * Fraction(2) ** (Ef - p["bias"])
    return -v if sign else v
