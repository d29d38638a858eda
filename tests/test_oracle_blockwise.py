"""Pins of the oracle's blockwise quantize (CPU only).

The "blockwise" recipe is only named on "FP8 training for Flux models"
(Configuration > Key FP8 Parameters).  Reading: 1 x 128 blocks along the
contraction for activations and gradients, 128 x 128 blocks for weights,
each with the largest power-of-two scale that keeps its amax within the FP8
maximum.  Pinned by hand-worked codes, an exact restatement of the scale
choice with Python fractions plus the independent encoder, the
no-saturation / top-binade property, layout invariants, and the GEMM
identity sum_k a b X_A X_B = sum over 128-blocks of (partial sum) / (s_a s_b).
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import parse_value, read_golden
from fp8_ref import ref_encode
from test_oracle_mx import bf16_bits, bits_to_f64

FMT = {"e4m3fn": 0, "e5m2": 1}
FMAX = {0: 448.0, 1: 57344.0}


def test_codes_golden(orc):
    for name, amax, code, *_ in read_golden("blockwise_codes.txt"):
        assert orc.blockwise_code(parse_value(amax), FMT[name]) == int(code), (name, amax)
    assert orc.blockwise_code(float("nan"), 0) == 127
    assert orc.blockwise_code(float("inf"), 1) == 127


def ind_exp(amax, fmt):
    """Largest e with amax * 2^e <= fmax, by exact rational comparison."""
    if amax == 0 or not np.isfinite(amax):
        return 0
    a, fm = Fraction(amax), Fraction(FMAX[fmt])
    e = 0
    while a * Fraction(2) ** e > fm:
        e -= 1
    while a * Fraction(2) ** (e + 1) <= fm:
        e += 1
    return max(-127, min(127, e))


def _x(seed, shape=(256, 384)):
    g = np.random.default_rng(seed)
    x = g.standard_normal(shape) * np.exp2(g.integers(-20, 20, size=(shape[0], 1)))
    x[5, :128] = 0.0
    x[7, 130] = np.inf
    x[9, shape[1] - 84] = np.nan
    return bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("fmt", [0, 1])
def test_activation_blocks_brute_force(orc, fmt):
    bits = _x(fmt)
    out = orc.blockwise_quantize(bits, fmt, 1)
    xv = bits_to_f64(bits)
    rows, cols = xv.shape
    for r in range(rows):
        for cb in range(cols // 128):
            blk = xv[r, 128 * cb:128 * cb + 128]
            fin = np.isfinite(blk).all()
            e = ind_exp(np.abs(blk).max() if fin else np.nan, fmt)
            assert (out["s_row"][r, 4 * cb:4 * cb + 4] == 127 - e).all(), (r, cb)
            for i in range(0, 128, 7):
                v = blk[i]
                if np.isnan(v):
                    continue
                want = ref_encode(float(v) * 2.0 ** e if np.isfinite(v) else float(v) * 1e300, fmt)
                assert out["q_row"][r, 128 * cb + i] == want


@pytest.mark.parametrize("fmt", [0, 1])
def test_no_saturation_and_top_binade(orc, fmt):
    bits = bf16_bits((np.random.default_rng(4).standard_normal((128, 512)) * 3).astype(np.float32))
    out = orc.blockwise_quantize(bits, fmt, 1)
    dec = np.array([orc.fp8_decode(c, fmt) for c in range(256)])
    q = np.abs(dec[out["q_row"]]).reshape(128, 4, 128)
    assert q.max() <= FMAX[fmt]
    assert (q.max(axis=2) >= FMAX[fmt] / 2).all()          # the block maximum is not wasted


def test_weight_blocks_shared_by_both_layouts(orc):
    bits = _x(7, (256, 256))
    out = orc.blockwise_quantize(bits, 0, 128)
    assert np.array_equal(out["q_colT"], out["q_row"].T)
    for rb in range(2):
        for cb in range(2):
            code = out["s_row"][128 * rb, 4 * cb]
            assert (out["s_row"][128 * rb:128 * rb + 128, 4 * cb:4 * cb + 4] == code).all()
            assert (out["s_col"][128 * cb:128 * cb + 128, 4 * rb:4 * rb + 4] == code).all()


def test_activation_colwise_is_rowwise_of_transpose(orc):
    bits = _x(8, (256, 384))
    a = orc.blockwise_quantize(bits, 1, 1, layouts=2)
    b = orc.blockwise_quantize(np.ascontiguousarray(bits.T), 1, 1, layouts=1)
    assert np.array_equal(a["q_colT"], b["q_row"]) and np.array_equal(a["s_col"], b["s_row"])


def test_gemm_is_sum_of_block_partials(orc):
    g = np.random.default_rng(9)
    A = g.integers(0, 0x7E, size=(3, 256)).astype(np.uint8)
    B = g.integers(0, 0x7E, size=(2, 256)).astype(np.uint8)
    ca = g.integers(115, 135, size=(3, 2))                  # one code per 128-block
    cb = g.integers(115, 135, size=(2, 2))
    sA = np.repeat(ca, 4, axis=1).astype(np.uint8)
    sB = np.repeat(cb, 4, axis=1).astype(np.uint8)
    ref, _ = orc.mx_gemm(A, 0, sA, B, 0, sB)
    for m in range(3):
        for n in range(2):
            tot = Fraction(0)
            mag = Fraction(0)
            for kb in range(2):
                sc = Fraction(2) ** (int(ca[m, kb]) - 127) * Fraction(2) ** (int(cb[n, kb]) - 127)
                prods = [Fraction(orc.fp8_decode(int(A[m, k]), 0)) * Fraction(orc.fp8_decode(int(B[n, k]), 0))
                         for k in range(128 * kb, 128 * kb + 128)]
                tot += sum(prods) * sc
                mag += sum(abs(p) for p in prods) * sc
            assert abs(Fraction(ref[m, n]) - tot) <= mag * Fraction(1, 2 ** 50)   # fp64 accumulation
