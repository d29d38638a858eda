"""Pins of the oracle's quantize and GEMM (CPU only).

Quantize: brute force on tiny tensors against the independent encoder of
fp8_ref.py with amax / scale computed here element by element; the
tensorwise layouts are exact transposes of each other; a rowwise row (or
colwise column) scaled by 2^j keeps its bytes and scales scale_inv by 2^j;
grouped colwise padding and per-group scales.

GEMM: an exact reference built from integer arithmetic -- every FP8 value is a
dyadic rational, so sum_k a_k b_k is computed exactly as a Fraction -- plus
special cases (one-hot operands, K = 16, empty groups) and grouped GEMM equal
to a loop of dense GEMMs.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from fp8_ref import PARAMS, is_nan_code, ref_encode

FMAX = {f: p[3] for f, p in PARAMS.items()}


def bits(t):
    return synth.bf16_bits(t)


def as_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def ref_scale(amax, fmt, margin=0):
    amax = np.float32(amax)
    if not (amax > 0) or not np.isfinite(amax):
        s = np.float32(1.0)
    else:
        with np.errstate(over="ignore"):
            s = np.float32(np.float32(FMAX[fmt]) / amax) * np.float32(2.0 ** -margin)
        if np.isinf(s):
            s = np.finfo(np.float32).max
    return np.float32(s), np.float32(np.float32(1.0) / s)


def brute_cast(xf, s, fmt):
    with np.errstate(over="ignore"):
        p = (xf * np.float32(s)).astype(np.float32)
    return ref_encode(float(p), fmt)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("shape", [(13, 37), (1, 5), (32, 16)])
def test_rowwise_brute_force(orc, fmt, shape):
    g = torch.Generator().manual_seed(sum(shape) + fmt)
    x = (torch.randn(shape, generator=g) * 3).to(torch.bfloat16)
    xb = bits(x)
    xf = as_f32(xb)
    out = orc.quantize(xb, fmt, orc.ROWWISE, margin=1)
    R, C = shape
    for r in range(R):
        s, si = ref_scale(np.abs(xf[r]).max(), fmt, 1)
        assert out["scale_inv_row"][r] == si
        for c in range(C):
            assert out["q_row"][r, c] == brute_cast(xf[r, c], s, fmt)
    for c in range(C):
        s, si = ref_scale(np.abs(xf[:, c]).max(), fmt, 1)
        assert out["scale_inv_col"][c] == si
        for r in range(R):
            assert out["q_colT"][c, r] == brute_cast(xf[r, c], s, fmt)
    assert out["amax"] == np.abs(xf).max()


@pytest.mark.parametrize("fmt", [0, 1])
def test_tensorwise_and_delayed(orc, fmt):
    g = torch.Generator().manual_seed(3)
    x = (torch.randn((48, 80), generator=g) * 0.1).to(torch.bfloat16)
    xb = bits(x)
    xf = as_f32(xb)
    am = np.abs(xf).max()
    t = orc.quantize(xb, fmt, orc.TENSORWISE)
    s, si = ref_scale(am, fmt)
    assert t["scale_inv_row"][0] == si and t["scale_inv_col"][0] == si and t["amax"] == am
    assert np.array_equal(t["q_colT"], t["q_row"].T)
    for r in range(0, 48, 5):
        for c in range(0, 80, 3):
            assert t["q_row"][r, c] == brute_cast(xf[r, c], s, fmt)
    # delayed: stored scale, amax accumulates by max into the history slot
    d = orc.quantize(xb, fmt, orc.DELAYED, scale_in=np.float32(3.0), amax_io=np.float32(0.5))
    assert d["amax"] == max(np.float32(0.5), am)
    assert d["scale_inv_row"][0] == np.float32(1.0) / np.float32(3.0)
    assert np.array_equal(d["q_colT"], d["q_row"].T)
    for r in range(0, 48, 7):
        for c in range(80):
            assert d["q_row"][r, c] == brute_cast(xf[r, c], 3.0, fmt)
    d2 = orc.quantize(xb, fmt, orc.DELAYED, scale_in=np.float32(3.0), amax_io=np.float32(1e9))
    assert d2["amax"] == np.float32(1e9)


def test_rowwise_power_of_two_invariance(orc):
    g = torch.Generator().manual_seed(4)
    x = torch.randn((16, 64), generator=g).to(torch.bfloat16)
    base = orc.quantize(bits(x), 0, orc.ROWWISE)
    for j in (-3, 1, 4):
        y = x.clone()
        y[5] = (y[5].float() * 2.0 ** j).to(torch.bfloat16)       # exact in bf16
        o = orc.quantize(bits(y), 0, orc.ROWWISE)
        assert np.array_equal(o["q_row"][5], base["q_row"][5])
        assert o["scale_inv_row"][5] == np.float32(base["scale_inv_row"][5] * 2.0 ** j)
        y = x.clone()
        y[:, 9] = (y[:, 9].float() * 2.0 ** j).to(torch.bfloat16)
        o = orc.quantize(bits(y), 0, orc.ROWWISE)
        assert np.array_equal(o["q_colT"][9], base["q_colT"][9])
        assert o["scale_inv_col"][9] == np.float32(base["scale_inv_col"][9] * 2.0 ** j)


def test_grouped_colwise_layout(orc):
    sizes = [5, 0, 33, 1, 0, 40]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    poff = orc.padded_offsets(off)
    assert list(poff) == [0, 32, 32, 96, 128, 128, 192]
    g = torch.Generator().manual_seed(9)
    x = torch.randn((int(off[-1]), 24), generator=g).to(torch.bfloat16)
    xb = bits(x)
    xf = as_f32(xb)
    o = orc.quantize(xb, 1, orc.ROWWISE, offsets=off)
    qT, sc = o["q_colT"], o["scale_inv_col"]
    assert qT.shape == (24, 192) and sc.shape == (6, 24)
    for e, m in enumerate(sizes):
        r0 = off[e]
        for c in range(24):
            if m == 0:
                assert sc[e, c] == 1.0
                continue
            s, si = ref_scale(np.abs(xf[r0:r0 + m, c]).max(), 1)
            assert sc[e, c] == si
            for r in range(m):
                assert qT[c, poff[e] + r] == brute_cast(xf[r0 + r, c], s, 1)
            assert not qT[c, poff[e] + m:poff[e + 1]].any()   # zero padding
    # rowwise part is unaffected by grouping
    o2 = orc.quantize(xb, 1, orc.ROWWISE)
    assert np.array_equal(o["q_row"], o2["q_row"])


def test_special_inputs(orc):
    vals = torch.tensor([[0.0, -0.0, float("inf"), 1.0],
                         [float("nan"), 2.0, -3.0, 1e-40],
                         [0.0, 0.0, 0.0, 0.0]], dtype=torch.float32).to(torch.bfloat16)
    o = orc.quantize(bits(vals), 0, orc.ROWWISE)
    assert o["scale_inv_row"][0] == 1.0          # Inf amax -> scale 1
    assert o["scale_inv_row"][1] == 1.0          # NaN amax -> scale 1
    assert o["scale_inv_row"][2] == 1.0          # all-zero row -> scale 1
    assert o["q_row"][0, 2] == 0x7E              # Inf saturates
    assert o["q_row"][0, 1] == 0x80              # -0 keeps its sign
    assert is_nan_code(int(o["q_row"][1, 0]), 0)
    assert np.isnan(o["amax"])


# --- GEMM ------------------------------------------------------------------

def exact_values(fmt):
    """Code -> exact Fraction, built from the bit fields (independent of the oracle)."""
    eb, mb, bias, _ = PARAMS[fmt]
    out = []
    for c in range(256):
        e = (c >> mb) & ((1 << eb) - 1)
        m = c & ((1 << mb) - 1)
        if e == 0:
            v = Fraction(m, 2 ** mb) * Fraction(2) ** (1 - bias)
        else:
            v = (1 + Fraction(m, 2 ** mb)) * Fraction(2) ** (e - bias)
        out.append(-v if c & 0x80 else v)
    return out


def finite_codes(rng, shape, fmt):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    bad = np.vectorize(lambda v: is_nan_code(int(v), fmt) or (fmt == 1 and (int(v) & 0x7F) == 0x7C), otypes=[bool])(c)
    c[bad] = 0x11
    return c


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_gemm_exact_bruteforce(orc, fa, fb):
    rng = np.random.default_rng(fa * 2 + fb)
    M, N, K = 7, 5, 48
    A = finite_codes(rng, (M, K), fa)
    B = finite_codes(rng, (N, K), fb)
    sa = rng.uniform(0.01, 2, size=M).astype(np.float32)
    sb = rng.uniform(0.01, 2, size=N).astype(np.float32)
    ref, bound = orc.gemm(A, fa, B, fb, sa, sb)
    va, vb = exact_values(fa), exact_values(fb)
    for m in range(M):
        for n in range(N):
            acc = sum(va[A[m, k]] * vb[B[n, k]] for k in range(K))
            absacc = sum(abs(va[A[m, k]] * vb[B[n, k]]) for k in range(K))
            ex = acc * Fraction(float(sa[m])) * Fraction(float(sb[n]))
            exb = absacc * abs(Fraction(float(sa[m])) * Fraction(float(sb[n])))
            assert abs(Fraction(ref[m, n]) - ex) <= Fraction(1, 10 ** 12) * (exb + 1)
            assert abs(Fraction(bound[m, n]) - exb) <= Fraction(1, 10 ** 12) * (exb + 1)


def test_gemm_special_cases(orc):
    K = 16
    A = np.zeros((4, K), np.uint8)
    for i in range(4):
        A[i, i] = 0x38                               # one-hot rows of 1.0 (e4m3)
    rng = np.random.default_rng(1)
    B = finite_codes(rng, (6, K), 0)
    ref, _ = orc.gemm(A, 0, B, 0, np.float32(2.0), np.float32(0.5))
    dec = np.array([orc.fp8_decode(c, 0) for c in range(256)])
    assert np.array_equal(ref, dec[B[:, :4]].T)      # picks column i of B, scale 2 * 0.5
    # scalar versus vector scales
    r1, _ = orc.gemm(B, 0, B, 0, np.float32(3.0), np.float32(0.25))
    r2, _ = orc.gemm(B, 0, B, 0, np.full(6, 3.0, np.float32), np.full(6, 0.25, np.float32))
    assert np.array_equal(r1, r2)
    # sampled points equal the full result
    pm = np.array([0, 5, 3]); pn = np.array([1, 0, 3])
    r3, _ = orc.gemm(B, 0, B, 0, np.float32(3.0), np.float32(0.25), points=(pm, pn))
    assert np.array_equal(r3, r1[pm, pn])


def test_grouped_gemm_equals_dense_loop(orc):
    rng = np.random.default_rng(2)
    sizes = [3, 0, 9, 1]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt, N, K, G = int(off[-1]), 6, 32, 4
    A = finite_codes(rng, (Mt, K), 0)
    B = finite_codes(rng, (G, N, K), 0)
    sa = rng.uniform(0.5, 2, size=Mt).astype(np.float32)
    sb = rng.uniform(0.5, 2, size=(G, N)).astype(np.float32)
    pm, pn = np.meshgrid(np.arange(Mt), np.arange(N), indexing="ij")
    ref, _ = orc.grouped_gemm(0, A, 0, B, 0, off, N, K, sa, sb.ravel(), None, pm.ravel(), pn.ravel())
    ref = ref.reshape(Mt, N)
    for e in range(G):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        d, _ = orc.gemm(A[r0:r1], 0, B[e], 0, sa[r0:r1], sb[e])
        assert np.array_equal(ref[r0:r1], d)
    # K_GROUPED: contraction over each group's rows in the padded colwise layout
    poff = orc.padded_offsets(off)
    ldT = int(poff[-1])
    Nk, Kk = 5, 7
    AT = np.zeros((Nk, ldT), np.uint8)
    BT = np.zeros((Kk, ldT), np.uint8)
    for e in range(G):
        m = sizes[e]
        AT[:, poff[e]:poff[e] + m] = finite_codes(rng, (Nk, m), 1)
        BT[:, poff[e]:poff[e] + m] = finite_codes(rng, (Kk, m), 0)
    sa2 = rng.uniform(0.5, 2, size=(G, Nk)).astype(np.float32)
    sb2 = rng.uniform(0.5, 2, size=(G, Kk)).astype(np.float32)
    pg, pn2, pk2 = np.meshgrid(np.arange(G), np.arange(Nk), np.arange(Kk), indexing="ij")
    ref2, _ = orc.grouped_gemm(1, AT, 1, BT, 0, off, Nk, Kk, sa2.ravel(), sb2.ravel(),
                               pg.ravel(), pn2.ravel(), pk2.ravel())
    ref2 = ref2.reshape(G, Nk, Kk)
    for e in range(G):
        m = sizes[e]
        if m == 0:
            assert not ref2[e].any()
            continue
        d, _ = orc.gemm(AT[:, poff[e]:poff[e] + m], 1, BT[:, poff[e]:poff[e] + m], 0, sa2[e], sb2[e])
        assert np.array_equal(ref2[e], d)


def test_results_do_not_depend_on_thread_count(orc):
    """The oracle parallelises only independent outer loops: one thread and
    several give the same bytes, scales and GEMM values bit for bit."""
    import oracle as oracle_mod
    g = torch.Generator().manual_seed(12)
    x = synth.bf16_bits((torch.randn((300, 264), generator=g) * 3).to(torch.bfloat16))
    xm = synth.bf16_bits((torch.randn((320, 256), generator=g) * 3).to(torch.bfloat16))  # MX: multiples of 32
    A = torch.randint(0, 0x7E, (40, 96), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    B = torch.randint(0, 0x7E, (56, 96), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    sa = (torch.rand(40, generator=g) + 0.5).numpy().astype(np.float32)
    sb = (torch.rand(56, generator=g) + 0.5).numpy().astype(np.float32)
    outs = []
    try:
        for threads in (1, 4):
            oracle_mod.set_threads(threads)
            q = orc.quantize(x, 0, orc.ROWWISE)
            mxq = orc.mx_quantize(xm, 1)
            ref, bound = orc.gemm(A, 0, B, 1, sa, sb)
            outs.append((q, mxq, ref, bound))
    finally:
        oracle_mod.set_threads(len(os.sched_getaffinity(0)))
    (q1, m1, r1, b1), (q4, m4, r4, b4) = outs
    for d1, d4 in ((q1, q4), (m1, m4)):
        for k in d1:
            assert np.asarray(d1[k]).tobytes() == np.asarray(d4[k]).tobytes(), k   # bit for bit
    assert r1.tobytes() == r4.tobytes() and b1.tobytes() == b4.tobytes()
