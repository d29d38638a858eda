"""Pins of the oracle's MXFP8 functions (CPU only).

MXFP8 is the "mxfp8" recipe of "FP8 training for Flux models"
(Configuration > Key FP8 Parameters) and the MXFP8 grouped GEMM that "FP8
Training on AMD GPUs with TorchTitan and TorchAO" names as next work.  The
pages give no definition; the oracle follows the OCP Microscaling v1.0
definition (blocks of 32, E8M0 scale 2^(floor(log2 amax) - emax_elem)).
Pinned here by:
  * hand-worked scale codes and blocks (golden fixtures);
  * a brute-force restatement per block that finds the scale by searching
    powers of two (no frexp) and encodes with the independent encoder of
    tests/fp8_ref.py;
  * reduction to the tensorwise oracle when every block has the same
    power-of-two amax;
  * layout invariants (colwise = rowwise of the transpose; grouped = the
    ungrouped quantize of each group, zero padding);
  * the dequantisation error bound;
  * the GEMM: exact rational arithmetic on tiny matrices, reduction to the
    per-tensor GEMM when every block scale is equal, and numpy's matmul of
    the dequantised operands.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import parse_value, read_golden
from fp8_ref import ref_encode

FMT = {"e4m3fn": 0, "e5m2": 1}
EMAX = {0: 8, 1: 15}
MAXV = {0: 448.0, 1: 57344.0}


def bf16_bits(vals) -> np.ndarray:
    t = torch.as_tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def is_nan_code(c, fmt):
    return (c & 0x7F) == 0x7F if fmt == 0 else (c & 0x7F) > 0x7C


# --- independent per-block restatement -------------------------------------

def ind_scale_exp(amax: float, fmt: int):
    """Largest e in [-127, 127] with 2^(e + emax) <= amax (searched, no frexp)."""
    if not math.isfinite(amax):
        return None
    e = -127
    while e < 127 and math.ldexp(1.0, e + 1 + EMAX[fmt]) <= amax:
        e += 1
    return e


def ind_block(vals, fmt):
    vals = [float(v) for v in vals]
    if any(not math.isfinite(v) for v in vals):
        return 255, None
    e = ind_scale_exp(max(abs(v) for v in vals), fmt)
    return e + 127, [ref_encode(v * 2.0 ** (-e), fmt) for v in vals]


# --- golden ---------------------------------------------------------------

def test_scale_codes_golden(orc):
    rows = read_golden("mx_scale_codes.txt")
    assert len(rows) >= 15
    for name, amax, code, *_ in rows:
        a = float(amax) if amax in ("inf", "nan") else parse_value(amax)
        assert orc.mx_scale_code(a, FMT[name]) == int(code), (name, amax)


def test_worked_blocks_golden(orc):
    for name, scale, vals, codes in read_golden("mx_worked_blocks.txt"):
        fmt = FMT[name]
        v = [parse_value(t) for t in vals.split(",")]
        x = np.zeros((1, 32), np.float32)
        x[0, :len(v)] = v
        out = orc.mx_quantize(bf16_bits(x), fmt, layouts=1)
        assert int(out["s_row"][0, 0]) == int(scale), name
        exp = [int(c, 16) for c in codes.split(",")]
        assert [int(c) for c in out["q_row"][0, :len(v)]] == exp, (name, vals)
        assert not out["q_row"][0, len(v):].any()


def test_e8m0_decode(orc):
    assert orc.e8m0_decode(127) == 1.0
    assert orc.e8m0_decode(0) == 2.0 ** -127
    assert orc.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(orc.e8m0_decode(255))


# --- brute force ----------------------------------------------------------

def _mx_inputs(seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((64, 256)).astype(np.float32)
    x[:8] *= np.exp2(g.integers(-140, 120, size=(8, 1))).astype(np.float32)   # tiny .. huge rows
    x[8:16] = g.lognormal(0, 6, size=(8, 256)).astype(np.float32) * g.choice([-1, 1], size=(8, 256))
    x[16, :32] = 0.0                                   # an all-zero block
    x[17, 5] = np.inf                                  # non-finite blocks
    x[18, 40] = np.nan
    x[19, 64:96] = 448.0 * 1.1                          # saturating block
    x[20, 96:128] = np.float32(2.0 ** -133)            # bf16 subnormals
    with np.errstate(over="ignore"):
        return bf16_bits(x)


@pytest.mark.parametrize("fmt", [0, 1])
def test_blocks_match_independent(orc, fmt):
    bits = _mx_inputs(fmt)
    out = orc.mx_quantize(bits, fmt, layouts=3)
    xv = bits_to_f64(bits)
    for r in range(xv.shape[0]):
        for b in range(xv.shape[1] // 32):
            code, q = ind_block(xv[r, 32 * b:32 * b + 32], fmt)
            assert out["s_row"][r, b] == code, (r, b)
            got = out["q_row"][r, 32 * b:32 * b + 32]
            if q is None:
                assert all(is_nan_code(int(c), fmt) for c in got)
            else:
                assert [int(c) for c in got] == q, (r, b)
    # colwise blocks run down the columns
    for c in range(0, xv.shape[1], 7):
        for b in range(xv.shape[0] // 32):
            code, q = ind_block(xv[32 * b:32 * b + 32, c], fmt)
            assert out["s_col"][c, b] == code
            got = out["q_colT"][c, 32 * b:32 * b + 32]
            if q is None:
                assert all(is_nan_code(int(v), fmt) for v in got)
            else:
                assert [int(v) for v in got] == q


@pytest.mark.parametrize("fmt", [0, 1])
def test_reduces_to_tensorwise_power_of_two(orc, fmt):
    """Every block's amax equal to the same 2^k: MX = tensorwise with the
    stored scale 2^(emax - k)."""
    g = np.random.default_rng(5 + fmt)
    k = 3
    x = (g.uniform(-1, 1, size=(32, 128)) * 2.0 ** k).astype(np.float32)
    x[:, ::32] = 2.0 ** k                              # each row block's amax
    x[::32, :] = 2.0 ** k                              # ... and each column block's
    bits = bf16_bits(x)
    mx = orc.mx_quantize(bits, fmt, layouts=3)
    assert (mx["s_row"] == k - EMAX[fmt] + 127).all()
    assert (mx["s_col"] == k - EMAX[fmt] + 127).all()
    tw = orc.quantize(bits, fmt, 0, layouts=3, scale_in=np.float32(2.0 ** (EMAX[fmt] - k)))
    assert np.array_equal(mx["q_row"], tw["q_row"])
    assert np.array_equal(mx["q_colT"], tw["q_colT"])


# --- layouts --------------------------------------------------------------

def test_colwise_is_rowwise_of_transpose(orc):
    bits = _mx_inputs(9)
    a = orc.mx_quantize(bits, 0, layouts=2)
    b = orc.mx_quantize(np.ascontiguousarray(bits.T), 0, layouts=1)
    assert np.array_equal(a["q_colT"], b["q_row"])
    assert np.array_equal(a["s_col"], b["s_row"])


@pytest.mark.parametrize("align", [32, 128])
def test_grouped_is_per_group_quantize(orc, align):
    sizes = [5, 0, 70, 1, 0, 129, 32]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    g = np.random.default_rng(11)
    x = g.standard_normal((int(off[-1]), 96)).astype(np.float32) * np.exp2(g.integers(-4, 4, size=(int(off[-1]), 1)))
    bits = bf16_bits(x)
    out = orc.mx_quantize(bits, 1, layouts=3, offsets=off, align=align)
    poff = orc.padded_offsets_align(off, align)
    assert out["q_colT"].shape == (96, int(poff[-1]))
    for e in range(len(sizes)):
        m = sizes[e]
        pad = int(poff[e + 1] - poff[e])
        assert pad == -(-m // align) * align
        blk = np.zeros((-(-m // 32) * 32, 96), np.uint16)
        blk[:m] = bits[off[e]:off[e + 1]]
        if blk.shape[0]:
            ref = orc.mx_quantize(blk, 1, layouts=3)
            got = out["q_colT"][:, poff[e]:poff[e] + blk.shape[0]]
            assert np.array_equal(got, ref["q_colT"])
            assert np.array_equal(out["s_col"][:, poff[e] // 32:poff[e] // 32 + blk.shape[0] // 32], ref["s_col"])
            assert np.array_equal(out["s_row"][poff[e]:poff[e] + m], ref["s_row"][:m])
            assert np.array_equal(out["q_row"][off[e]:off[e + 1]], ref["q_row"][:m])
        # padding: zero bytes, code 0
        assert not out["q_colT"][:, poff[e] + blk.shape[0]:poff[e + 1]].any()
        assert not out["s_col"][:, (poff[e] + blk.shape[0]) // 32:poff[e + 1] // 32].any()
        assert not out["s_row"][poff[e] + m:poff[e + 1]].any()


@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantisation_error_bound(orc, fmt):
    bits = _mx_inputs(20 + fmt)
    out = orc.mx_quantize(bits, fmt, layouts=1)
    dec = np.array([orc.fp8_decode(c, fmt) for c in range(256)])
    xv = bits_to_f64(bits)
    mb = 3 if fmt == 0 else 2
    for r in range(xv.shape[0]):
        for b in range(xv.shape[1] // 32):
            v = xv[r, 32 * b:32 * b + 32]
            code = int(out["s_row"][r, b])
            if code == 255:
                continue
            X = 2.0 ** (code - 127)
            q = dec[out["q_row"][r, 32 * b:32 * b + 32]]
            assert np.abs(q).max() <= MAXV[fmt]
            if code > 0 and np.abs(v).max() > 0:        # not clamped: the top element sits in the top binade
                assert np.abs(q).max() >= 2.0 ** EMAX[fmt]
            for vi, qi in zip(v, q):
                a = abs(vi) / X
                if a > MAXV[fmt]:
                    assert abs(qi) == MAXV[fmt]
                else:
                    ulp = 2.0 ** (max(math.frexp(a)[1] - 1, 1 - (7 if fmt == 0 else 15)) - mb) if a > 0 else 0
                    assert abs(qi * X - vi) <= 0.5 * ulp * X + 1e-300


# --- GEMM -----------------------------------------------------------------

def _codes(g, shape, fmt):
    c = g.integers(0, 256, size=shape).astype(np.uint8)
    nanm = (c & 0x7F) == 0x7F if fmt == 0 else (c & 0x7F) >= 0x7C
    c[nanm] = 0x38 if fmt == 0 else 0x3C
    return c


def test_gemm_exact_rational(orc):
    g = np.random.default_rng(3)
    M, N, K = 3, 2, 96
    A, B = _codes(g, (M, K), 0), _codes(g, (N, K), 1)
    sA = g.integers(110, 140, size=(M, K // 32)).astype(np.uint8)
    sB = g.integers(110, 140, size=(N, K // 32)).astype(np.uint8)
    ref, bound = orc.mx_gemm(A, 0, sA, B, 1, sB)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            ab = Fraction(0)
            for k in range(K):
                p = (Fraction(orc.fp8_decode(int(A[m, k]), 0)) * Fraction(orc.fp8_decode(int(B[n, k]), 1))
                     * Fraction(2) ** (int(sA[m, k // 32]) - 127) * Fraction(2) ** (int(sB[n, k // 32]) - 127))
                acc += p
                ab += abs(p)
            assert abs(Fraction(ref[m, n]) - acc) <= ab * Fraction(1, 2 ** 50)
            assert abs(Fraction(bound[m, n]) - ab) <= ab * Fraction(1, 2 ** 50)


def test_gemm_uniform_scales_equal_tensor_gemm(orc):
    g = np.random.default_rng(4)
    M, N, K = 17, 9, 160
    A, B = _codes(g, (M, K), 0), _codes(g, (N, K), 0)
    sA = np.full((M, K // 32), 120, np.uint8)
    sB = np.full((N, K // 32), 131, np.uint8)
    ref, bound = orc.mx_gemm(A, 0, sA, B, 0, sB)
    r2, b2 = orc.gemm(A, 0, B, 0, np.float32(2.0 ** -7), np.float32(2.0 ** 4))
    assert np.array_equal(ref, r2) and np.array_equal(bound, b2)


def test_gemm_matches_numpy_dequantised(orc):
    g = np.random.default_rng(6)
    M, N, K = 40, 24, 256
    A, B = _codes(g, (M, K), 0), _codes(g, (N, K), 1)
    sA = g.integers(100, 150, size=(M, K // 32)).astype(np.uint8)
    sB = g.integers(100, 150, size=(N, K // 32)).astype(np.uint8)
    ta = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    da = ta.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    db = ta.view(torch.float8_e5m2).to(torch.float64).numpy()
    Ad = da[A] * np.repeat(np.exp2(sA.astype(np.float64) - 127), 32, axis=1)
    Bd = db[B] * np.repeat(np.exp2(sB.astype(np.float64) - 127), 32, axis=1)
    ref, bound = orc.mx_gemm(A, 0, sA, B, 1, sB)
    want = Ad @ Bd.T
    assert np.all(np.abs(ref - want) <= 1e-12 * (np.abs(Ad) @ np.abs(Bd).T) + 1e-300)
    pts = (g.integers(0, M, 50), g.integers(0, N, 50))
    rp, bp = orc.mx_gemm(A, 0, sA, B, 1, sB, points=pts)
    assert np.array_equal(rp, ref[pts]) and np.array_equal(bp, bound[pts])
