"""Pins of the oracle's scale formula and amax-history update (CPU only).

Pinned against: hand-worked fp32 scales (golden), a hand-stepped L = 4
history sequence (golden), and the invariants that the recipe's definitions
imply (window contents, most_recent vs max, margin as an exact power of two,
L = 1 making the two algorithms equal, non-finite amax handling).
"""
import math

import numpy as np
import pytest

from conftest import parse_value, read_golden

FMT = {"e4m3fn": 0, "e5m2": 1, "e4m3fnuz": 2}
FMAX = {0: 448.0, 1: 57344.0, 2: 240.0}


def f32hex(x):
    return format(int(np.float32(x).view(np.uint32)), "08x")


def test_scale_worked_examples(orc):
    rows = read_golden("scale_worked_examples.txt")
    assert len(rows) == 6
    for name, amax, margin, s_hex, si_hex in rows:
        s, si = orc.current_scale(parse_value(amax), FMT[name], int(margin))
        assert f32hex(s) == s_hex, (name, amax, margin)
        assert f32hex(si) == si_hex, (name, amax, margin)


def test_scale_special_amax(orc):
    for amax in (0.0, float("inf"), float("nan")):
        s, si = orc.current_scale(amax, 0, 0)
        assert s == 1.0 and si == 1.0
    # tiny amax: 448 / 1e-45 overflows fp32 -> FLT_MAX
    s, si = orc.current_scale(1e-45, 0, 0)
    assert s == np.finfo(np.float32).max
    assert si == np.float32(1.0) / np.finfo(np.float32).max


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_margin_is_exact_power_of_two(orc, fmt):
    rng = np.random.default_rng(fmt)
    for amax in rng.uniform(1e-3, 1e3, size=200).astype(np.float32):
        s0, _ = orc.current_scale(amax, fmt, 0)
        for m in (1, 2, 5):
            sm, sim = orc.current_scale(amax, fmt, m)
            assert sm == np.float32(s0 * 2.0 ** -m)
            assert sim == np.float32(1.0) / sm


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_scaled_amax_lands_on_max(orc, fmt):
    """amax * scale encodes to the largest code (or its neighbour below) and never above max."""
    rng = np.random.default_rng(7)
    top = orc.fp8_max_code(fmt)
    for amax in rng.lognormal(0, 4, size=300).astype(np.float32):
        s, _ = orc.current_scale(amax, fmt, 0)
        p = np.float32(amax * s)
        code = orc.fp8_encode(float(p), fmt)
        assert orc.fp8_decode(code, fmt) <= FMAX[fmt]
        assert code in (top, top - 1)


def _run_history(orc, amaxes, L, algo, margin=0, fmt=0):
    hist = np.zeros((1, L), np.float32)
    scale = np.ones(1, np.float32)
    sinv = np.ones(1, np.float32)
    cnt = np.zeros(1, np.int32)
    out = []
    for a in amaxes:
        hist[0, 0] = max(hist[0, 0], np.float32(a)) if not math.isnan(a) else np.float32("nan")
        orc.update_amax_history(hist, scale, sinv, fmt, algo, margin, cnt)
        out.append((scale[0], sinv[0], hist.copy(), cnt[0]))
    return out


def test_history_l4_table(orc):
    rows = read_golden("history_l4.txt")
    amaxes = [float(r[1]) for r in rows]
    mr = _run_history(orc, amaxes, 4, orc.MOST_RECENT)
    mx = _run_history(orc, amaxes, 4, orc.MAX)
    for (step, a, d_mr, d_mx), r_mr, r_mx in zip(rows, mr, mx):
        assert r_mr[0] == np.float32(448.0) / np.float32(float(d_mr)), step
        assert r_mx[0] == np.float32(448.0) / np.float32(float(d_mx)), step
        assert r_mx[1] == np.float32(1.0) / r_mx[0]


def test_history_window_invariants(orc):
    rng = np.random.default_rng(11)
    L = 8
    amaxes = rng.lognormal(0, 1, size=20).astype(np.float32)
    res = _run_history(orc, amaxes, L, orc.MAX)
    for k, (s, si, hist, _) in enumerate(res, start=1):
        h = hist[0]
        assert h[0] == 0.0                      # current slot cleared after the update
        assert np.count_nonzero(h) <= k          # never more entries than steps
        n = min(k, L - 1)
        # newest first: H[1..n] are the last n amaxes
        assert np.array_equal(h[1:n + 1], amaxes[k - n:k][::-1])
        # the scale used the window of the current and previous L-1 amaxes
        win = amaxes[max(0, k - L):k]
        assert s == np.float32(448.0) / np.float32(win.max())


def test_max_is_more_conservative(orc):
    rng = np.random.default_rng(5)
    amaxes = rng.lognormal(0, 1, size=40).astype(np.float32)
    mr = _run_history(orc, amaxes, 16, orc.MOST_RECENT)
    mx = _run_history(orc, amaxes, 16, orc.MAX)
    for a, b in zip(mr, mx):
        assert b[0] <= a[0]


def test_l1_algos_identical(orc):
    rng = np.random.default_rng(6)
    amaxes = rng.lognormal(0, 2, size=30).astype(np.float32)
    mr = _run_history(orc, amaxes, 1, orc.MOST_RECENT)
    mx = _run_history(orc, amaxes, 1, orc.MAX)
    for a, b in zip(mr, mx):
        assert a[0] == b[0] and a[1] == b[1]


def test_most_recent_ignores_older_entries(orc):
    hist = np.zeros((2, 5), np.float32)
    hist[0] = [2.0, 100.0, 100.0, 100.0, 100.0]
    hist[1] = [2.0, 0.0, 0.0, 0.0, 0.0]
    scale = np.ones(2, np.float32)
    sinv = np.ones(2, np.float32)
    orc.update_amax_history(hist, scale, sinv, 0, orc.MOST_RECENT, 0)
    assert scale[0] == scale[1] == np.float32(224.0)


def test_margin_in_update(orc):
    for m in range(4):
        hist = np.array([[3.0, 0.0]], np.float32)
        scale = np.ones(1, np.float32)
        sinv = np.ones(1, np.float32)
        orc.update_amax_history(hist, scale, sinv, 0, orc.MOST_RECENT, m)
        assert scale[0] == np.float32(np.float32(448.0) / np.float32(3.0)) * np.float32(2.0 ** -m)


def test_nonfinite_and_zero_keep_scale(orc):
    hist = np.zeros((4, 3), np.float32)
    hist[:, 0] = [np.inf, np.nan, 0.0, 4.0]
    scale = np.full(4, 7.0, np.float32)
    sinv = np.full(4, 0.5, np.float32)
    cnt = np.zeros(4, np.int32)
    orc.update_amax_history(hist, scale, sinv, np.array([0, 1, 0, 1], np.uint8), orc.MOST_RECENT, 0, cnt)
    assert list(scale[:3]) == [7.0, 7.0, 7.0] and list(sinv[:3]) == [0.5, 0.5, 0.5]
    assert list(cnt) == [1, 1, 0, 0]
    assert scale[3] == np.float32(57344.0 / 4.0)
    # NaN anywhere in a max window propagates
    hist = np.array([[1.0, np.nan, 2.0]], np.float32)
    scale = np.full(1, 3.0, np.float32)
    sinv = np.full(1, 1 / 3, np.float32)
    cnt = np.zeros(1, np.int32)
    orc.update_amax_history(hist, scale, sinv, 0, orc.MAX, 0, cnt)
    assert scale[0] == np.float32(3.0) and cnt[0] == 1
    assert hist[0, 0] == 0.0 and hist[0, 1] == 1.0 and np.isnan(hist[0, 2])


def test_per_tensor_format(orc):
    hist = np.array([[2.0, 0], [2.0, 0], [2.0, 0]], np.float32)
    scale = np.ones(3, np.float32)
    sinv = np.ones(3, np.float32)
    orc.update_amax_history(hist, scale, sinv, np.array([0, 1, 2], np.uint8), orc.MOST_RECENT, 0)
    assert list(scale) == [224.0, 28672.0, 120.0]
