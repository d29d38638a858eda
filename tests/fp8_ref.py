"""Independent FP8 reference encoder used by the oracle's pin tests.

Written in plain arithmetic on Python floats (frexp, round-half-even), not
bit manipulation, so that it shares no method with the oracle's table search.
Format parameters are the OCP 8-bit float definitions; maxima 448 / 240 are
the ones printed on "FP8 Training on MI300X" ("Discovered AMD FP8 dtype
difference").  The fnuz formats (e4m3fnuz, e5m2fnuz, named on the same page)
reserve no exponent for Inf/NaN, take bias + 1, use 0x80 as their only NaN
and have no negative zero.
"""
import math

PARAMS = {  # exponent bits, mantissa bits, bias, max
    0: (4, 3, 7, 448.0),     # e4m3fn
    1: (5, 2, 15, 57344.0),  # e5m2
    2: (4, 3, 8, 240.0),     # e4m3fnuz
    3: (5, 2, 16, 57344.0),  # e5m2fnuz
}
FNUZ = (2, 3)


def is_nan_code(c, fmt):
    if fmt in FNUZ:
        return c == 0x80
    if fmt == 0:
        return (c & 0x7F) == 0x7F
    return (c & 0x7F) > 0x7C


def is_inf_code(c, fmt):
    return fmt == 1 and (c & 0x7F) == 0x7C


def _value_to_code_table(fmt):
    """Map exact value -> code, built by brute force from decode formulas
    written independently here (value = (1 + m/2^mb) 2^(e-bias) or subnormal)."""
    eb, mb, bias, _ = PARAMS[fmt]
    table = {}
    for c in range(256):
        if is_nan_code(c, fmt) or is_inf_code(c, fmt):
            continue
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> mb) & ((1 << eb) - 1)
        m = c & ((1 << mb) - 1)
        v = (m / 2 ** mb) * 2.0 ** (1 - bias) if e == 0 else (1 + m / 2 ** mb) * 2.0 ** (e - bias)
        v = s * v
        if v == 0 and fmt in FNUZ:
            table[0.0] = 0
            continue
        key = (v, math.copysign(1.0, v))
        table[key] = c
    return table


_TABLES = {f: _value_to_code_table(f) for f in PARAMS}


def ref_encode(v: float, fmt: int) -> int:
    eb, mb, bias, vmax = PARAMS[fmt]
    if math.isnan(v):
        return -1  # NaN class
    sign = math.copysign(1.0, v)
    a = abs(v)
    if a >= vmax:
        mag = vmax
    elif a == 0.0:
        mag = 0.0
    else:
        _, ex = math.frexp(a)        # a = f * 2^ex, f in [0.5, 1)
        e = max(ex - 1, 1 - bias)    # binade exponent, clamped to the subnormal range
        ulp = 2.0 ** (e - mb)
        mag = round(a / ulp) * ulp   # a / ulp is exact; round() is ties-to-even
    if fmt in FNUZ:
        if mag == 0.0:
            return 0
        return _TABLES[fmt][(sign * mag, sign)]
    return _TABLES[fmt][(sign * mag, sign)]
