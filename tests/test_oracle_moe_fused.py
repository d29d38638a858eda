"""Pins of the oracle's MoE prologues (CPU only): the gather that permutes
token rows into expert order and SwiGLU, fused in front of the MX quantize
("FP8 Training on AMD GPUs with TorchTitan and TorchAO": a five-kernel eager
chain replaced by one fused kernel on the MoE path).

  * bf16_from_double against a brute-force nearest point of the finite bf16
    set (exact rationals, ties to the even code, overflow past the midpoint
    above the largest value) and against PyTorch's fp32 -> bf16 conversion on
    values that fp32 holds exactly;
  * SwiGLU h = bf16(silu(g) * u) against the correctly rounded result of a
    high-precision evaluation (mpmath, 80-bit significands): every finite bf16
    gate with u = 1, and random gate / up pairs over wide ranges;
  * its limits: silu(+Inf) = +Inf, silu(-Inf) = -0, exp(-g) underflow and
    overflow, NaN propagation, the sign of zero;
  * the gather: identity = plain quantize, a permutation permutes the row
    layout, repeated indices repeat rows.
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest
import torch

from test_oracle_mx import bf16_bits, bits_to_f64

# the finite non-negative bf16 values, ascending, with their codes
_CODES = np.arange(0, 0x7F80, dtype=np.uint16)
_VALS = [Fraction(float(v)) for v in torch.from_numpy(_CODES.view(np.int16)).view(torch.bfloat16).double().numpy()]
_TOP = Fraction(2) ** 128  # the next power of two above the largest value: the overflow point


def nearest_bf16(x) -> int:
    """Code of the bf16 value nearest to the exact rational x (ties to the
    even code; at or past the midpoint above the largest value: Inf)."""
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    i = bisect.bisect_left(_VALS, a)
    if i == len(_VALS):                       # above the largest finite value
        lo, hi = len(_VALS) - 1, None
    elif _VALS[i] == a:
        return sign | int(_CODES[i])
    else:
        lo, hi = i - 1, i
    vlo = _VALS[lo]
    vhi = _TOP if hi is None else _VALS[hi]
    dlo, dhi = a - vlo, vhi - a
    if dlo < dhi or (dlo == dhi and _CODES[lo] % 2 == 0):
        return sign | int(_CODES[lo])
    return sign | (0x7F80 if hi is None else int(_CODES[hi]))


def test_bf16_from_double_is_nearest(orc):
    g = np.random.default_rng(0)
    mags = np.exp2(g.uniform(-140, 129, size=6000))
    vals = list(mags * g.choice([-1.0, 1.0], size=mags.size))
    # exact midpoints between neighbours (ties), in the normal and subnormal ranges
    for k in g.integers(1, len(_VALS) - 1, size=1500):
        vals.append(float((_VALS[k] + _VALS[k + 1]) / 2))
    for k in range(1, 300):
        vals.append(float((_VALS[k] + _VALS[k + 1]) / 2))
    top = _VALS[-1]
    vals += [float((top + _TOP) / 2), float((top + _TOP) / 2) * (1 - 2 ** -40), 0.0, -0.0, 2.0 ** -134,
             2.0 ** -134 * (1 + 2 ** -30), 1e300, -1e300, 2.0 ** -1000]
    for v in vals:
        want = nearest_bf16(Fraction(v))
        if v == 0 and np.signbit(v):
            want = 0x8000
        assert orc.bf16_from_double(v) == want, (v, hex(orc.bf16_from_double(v)), hex(want))


def test_bf16_from_double_matches_torch_on_fp32(orc):
    g = np.random.default_rng(1)
    u = g.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    u[:2000] = (u[:2000] & 0xFFFF0000) | 0x8000        # exact ties
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_double(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)


def _mp_swiglu_bits(gb, ub):
    """Correctly rounded bf16(silu(g) * u) for finite g, u.

    With P = g u (exact), the product is P sigma(g), sigma(g) = 1 / (1 +
    e^-g).  Its bracket of bf16 neighbours comes from a 100-bit evaluation;
    the side of their midpoint M is the sign of d = P sigma(g) - M, taken
    from a form in which the exact rational part and the transcendental
    part (100-bit relative accuracy) do not cancel:
        |g| < 1 : d = (P / 2 - M) + (P / 2) tanh(g / 2)
        g >= 1  : d = (P - M) - P / (1 + e^g)
        g <= -1 : d = P / (1 + e^-g) - M
    """
    import mpmath
    mpmath.mp.prec = 100

    def frac(x):                      # an mpf as an exact rational
        if x == 0:
            return Fraction(0)
        man, exp = abs(x).man_exp
        f = Fraction(int(man)) * Fraction(2) ** int(exp)
        return -f if x < 0 else f

    out = np.zeros(gb.size, np.uint16)
    gv, uv = bits_to_f64(gb), bits_to_f64(ub)
    for i, (gd, ud) in enumerate(zip(gv, uv)):
        neg = bool(np.signbit(gd)) != bool(np.signbit(ud))   # sign of the product, of a zero too
        if gd == 0 or ud == 0:
            out[i] = 0x8000 if neg else 0
            continue
        g = mpmath.mpf(gd)
        P = Fraction(gd) * Fraction(ud)
        a = abs(g / (1 + mpmath.exp(-g)) * mpmath.mpf(ud))
        if a < mpmath.mpf(2) ** -140:            # below a quarter of the smallest bf16: a signed zero
            out[i] = 0x8000 if neg else 0
            continue
        if a > mpmath.mpf(2) ** 129:             # far past the overflow point
            out[i] = 0xFF80 if neg else 0x7F80
            continue
        k = bisect.bisect_left(_VALS, frac(a))
        lo = max(k - 1, 0)
        vlo = _VALS[lo]
        vhi = _VALS[lo + 1] if lo + 1 < len(_VALS) else _TOP
        M = (vlo + vhi) / 2 * (-1 if neg else 1)    # the signed midpoint
        Pm = mpmath.mpf(P.numerator) / P.denominator
        if abs(gd) < 1:
            R, T = P / 2 - M, Pm / 2 * mpmath.tanh(g / 2)
        elif gd >= 1:
            R, T = P - M, -Pm / (1 + mpmath.exp(g))
        else:
            R, T = -M, Pm / (1 + mpmath.exp(-g))
        # sign of d = R + T; a T far below |R| (e^-g for huge g) never becomes a rational
        if R == 0:
            d = 1 if T > 0 else -1
        elif abs(T) < abs(mpmath.mpf(R.numerator) / R.denominator) / 2:
            d = R
        else:
            d = R + frac(T)
        beyond = d > 0 if not neg else d < 0      # |product| above |M|
        assert d != 0 and T != 0
        if beyond:
            out[i] = 0x7F80 if lo + 1 == len(_VALS) else int(_CODES[lo + 1])
        else:
            out[i] = int(_CODES[lo])
        if neg:
            out[i] |= 0x8000
    return out


def test_swiglu_every_gate_value(orc):
    """All finite bf16 gate values with u = 1 and u = -0.75."""
    codes = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    finite = (codes & 0x7F80) != 0x7F80
    gb = codes[finite]
    for uval in (1.0, -0.75):
        ub = bf16_bits(np.full(gb.size, uval, np.float32))
        got = orc.swiglu_bf16(gb, ub)
        want = _mp_swiglu_bits(gb, ub)
        bad = got != want
        assert not bad.any(), (uval, int(bad.sum()), [hex(int(v)) for v in gb[bad][:5]])


def test_swiglu_random_pairs(orc):
    g = np.random.default_rng(2)
    n = 20000
    gv = (g.standard_normal(n) * 4).astype(np.float32)
    uv = (g.standard_normal(n) * np.exp2(g.uniform(-20, 20, size=n))).astype(np.float32)
    gb, ub = bf16_bits(gv), bf16_bits(uv)
    got = orc.swiglu_bf16(gb, ub)
    want = _mp_swiglu_bits(gb, ub)
    assert np.array_equal(got, want)


def test_swiglu_limits(orc):
    g = bf16_bits(np.array([0.0, 100.0, -100.0, 300.0, -300.0, float("nan"), 1.0, float("inf"), -float("inf"),
                            -float("inf"), float("inf")], np.float32))
    u = bf16_bits(np.array([3.0, 1.5, 2.0, -1.0, -2.0, 1.0, float("nan"), 2.0, 2.0, float("inf"), 0.0],
                           np.float32))
    h = bits_to_f64(orc.swiglu_bf16(g, u))
    assert h[0] == 0.0
    assert h[1] == 150.0                      # e^-100 is far below half an ulp of 1: silu(g) = g
    assert h[2] == 0.0 and np.signbit(h[2])   # silu(-100) * 2 = -7.4e-42, below the smallest bf16: -0
    assert h[3] == -300.0
    assert h[4] == 0.0 and not np.signbit(h[4])   # (-0) * (-2) = +0
    assert np.isnan(h[5]) and np.isnan(h[6])
    assert h[7] == float("inf")               # silu(+Inf) = +Inf
    assert h[8] == 0.0 and np.signbit(h[8])   # silu(-Inf) = -0 (the limit), times 2
    assert np.isnan(h[9])                     # -0 * Inf
    assert np.isnan(h[10])                    # Inf * 0


def test_gather_identity_and_permutation(orc):
    g = np.random.default_rng(2)
    x = bf16_bits((g.standard_normal((96, 160)) * np.exp2(g.integers(-5, 5, size=(96, 1)))).astype(np.float32))
    ident = orc.mx_permute_quantize(x, np.arange(96), 0, 1)
    plain = orc.mx_quantize(x, 0, 1)
    assert np.array_equal(ident["q_row"], plain["q_row"]) and np.array_equal(ident["s_row"], plain["s_row"])
    perm = g.permutation(96)
    out = orc.mx_permute_quantize(x, perm, 0, 1)
    assert np.array_equal(out["q_row"], plain["q_row"][perm])
    assert np.array_equal(out["s_row"], plain["s_row"][perm])
    rep = np.array([5, 5, 0, 95, 5] + list(range(27)), np.int64)      # a token routed to several experts
    out = orc.mx_permute_quantize(x, rep, 1, 1)
    ref = orc.mx_quantize(x, 1, 1)
    assert np.array_equal(out["q_row"], ref["q_row"][rep])


def test_swiglu_quantize_composition(orc):
    g = np.random.default_rng(3)
    gu = bf16_bits((g.standard_normal((64, 256)) * 3).astype(np.float32))
    out = orc.mx_swiglu_quantize(gu, 0, 3)
    h = orc.swiglu_bf16(gu[:, :128], gu[:, 128:])
    assert np.array_equal(out["h"], h)
    ref = orc.mx_quantize(h, 0, 3)
    for k in ("q_row", "s_row", "q_colT", "s_col"):
        assert np.array_equal(out[k], ref[k])


def test_rowwise_prologue_compositions(orc):
    """The rowwise prologues are compositions: the identity gather is the
    plain grouped quantize, a repeated index repeats a row (bytes and row
    scale), and the SwiGLU prologue quantizes the SwiGLU output."""
    g = np.random.default_rng(4)
    x = bf16_bits((g.standard_normal((96, 160)) * np.exp2(g.integers(-5, 5, size=(96, 1)))).astype(np.float32))
    off = np.array([0, 30, 30, 96], np.int32)
    ident = orc.permute_quantize(x, np.arange(96), 1, orc.ROWWISE, off)
    plain = orc.quantize(x, 1, orc.ROWWISE, offsets=off)
    for k in ("q_row", "scale_inv_row", "q_colT", "scale_inv_col"):
        assert np.array_equal(ident[k], plain[k])
    src = np.arange(96)
    src[10:20] = 7                                        # token 7 routed to ten experts' slots
    rep = orc.permute_quantize(x, src, 1, orc.ROWWISE, off)
    for r in range(10, 20):
        assert np.array_equal(rep["q_row"][r], rep["q_row"][7])
        assert rep["scale_inv_row"][r] == rep["scale_inv_row"][7]
    gu = bf16_bits((g.standard_normal((96, 256)) * 3).astype(np.float32))
    out = orc.swiglu_quantize(gu, 0, orc.ROWWISE, off)
    h = orc.swiglu_bf16(gu[:, :128], gu[:, 128:])
    assert np.array_equal(out["h"], h)
    ref = orc.quantize(h, 0, orc.ROWWISE, offsets=off)
    for k in ("q_row", "scale_inv_row", "q_colT", "scale_inv_col"):
        assert np.array_equal(out[k], ref[k])
