"""Pins of the oracle's FP8 codec (CPU only).

The codec is pinned against things other than itself:
  * the format maxima printed on the pages (golden fixture);
  * worked encodings derived by hand from the format definitions (golden);
  * exhaustive properties over all 256 codes (round trip, monotonicity);
  * a second encoder written here in plain float arithmetic (frexp / round),
    not bit manipulation;
  * PyTorch's own float8 casts (a library cross-check) on dense sweeps.
"""
import math

import numpy as np
import pytest
import torch

from conftest import parse_value, read_golden
from fp8_ref import PARAMS, is_inf_code, is_nan_code, ref_encode

FMT = {"e4m3fn": 0, "e5m2": 1, "e4m3fnuz": 2, "e5m2fnuz": 3}
TORCH_DT = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2, 2: torch.float8_e4m3fnuz,
            3: torch.float8_e5m2fnuz}
ALL_FMTS = [0, 1, 2, 3]
# --- tests -------------------------------------------------------------------

def test_maxima_match_pages(orc):
    for name, vmax, code in read_golden("fp8_format_maxima.txt"):
        f = FMT[name]
        assert orc.fp8_max_value(f) == float(vmax)
        assert orc.fp8_max_code(f) == int(code, 16)
        assert orc.fp8_decode(int(code, 16), f) == float(vmax)


def test_worked_codes(orc):
    rows = read_golden("fp8_worked_codes.txt")
    assert len(rows) >= 20
    for name, val, code, *_ in rows:
        f = FMT[name]
        assert orc.fp8_encode(parse_value(val), f) == int(code, 16), (name, val)


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_roundtrip_all_codes(orc, fmt):
    n_checked = 0
    for c in range(256):
        v = orc.fp8_decode(c, fmt)
        if is_nan_code(c, fmt):
            assert math.isnan(v)
            assert is_nan_code(orc.fp8_encode(v, fmt), fmt)
            continue
        if is_inf_code(c, fmt):
            assert math.isinf(v)
            # saturating cast: +-Inf goes to +-max
            assert orc.fp8_encode(v, fmt) == (c & 0x80) | orc.fp8_max_code(fmt)
            continue
        assert orc.fp8_encode(v, fmt) == c, hex(c)
        n_checked += 1
    assert n_checked == {0: 254, 1: 248, 2: 255, 3: 255}[fmt]


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_decode_strictly_monotone(orc, fmt):
    vals = [orc.fp8_decode(c, fmt) for c in range(orc.fp8_max_code(fmt) + 1)]
    assert vals[0] == 0.0
    assert all(b > a for a, b in zip(vals, vals[1:]))
    # negative half mirrors the positive half (fnuz: 0x80 is NaN instead of -0)
    for c in range(1, orc.fp8_max_code(fmt) + 1):
        assert orc.fp8_decode(0x80 | c, fmt) == -vals[c]


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_decode_matches_torch(orc, fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()
    for c in range(256):
        ov = orc.fp8_decode(c, fmt)
        if math.isnan(ov):
            assert math.isnan(tv[c])
        else:
            assert ov == tv[c], hex(c)


def _sweep_values():
    """Every bf16 bit pattern as fp32, times a grid of scales, plus random fp32."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    base = bits.view(np.float32)
    base = base[np.isfinite(base)]
    scales = np.array([1.0, 2.0 ** -7, 448.0 / 3.0, 0.7, 57344.0 / 9.5, 240.0 / 3.3], np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        vals = [(base * s).astype(np.float32) for s in scales]
    rng = np.random.default_rng(123)
    rnd = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    vals.append(rnd[np.isfinite(rnd)])
    return np.concatenate(vals)


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_encode_matches_torch_cast(orc, fmt):
    """torch's fp8 cast of clamp(v, -max, max) equals the saturating encode."""
    v = _sweep_values()
    vmax = PARAMS[fmt][3]
    # oracle codes for the whole sweep (cast_points with scale 1 takes bf16 input;
    # here inputs are fp32, so go through the scalar entry point on a subsample
    # and through torch for the full set)
    t = torch.from_numpy(np.clip(v, -vmax, vmax).astype(np.float32))
    tc = t.to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    rng = np.random.default_rng(fmt)
    idx = rng.choice(v.size, size=60_000, replace=False)
    for i in idx:
        oc = orc.fp8_encode(float(v[i]), fmt)
        if fmt in (2, 3) and oc == 0:
            assert tc[i] in (0x00,), (v[i], tc[i])
        else:
            assert oc == tc[i], (fmt, float(v[i]), hex(oc), hex(tc[i]))


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_encode_matches_independent_encoder(orc, fmt):
    v = _sweep_values()
    rng = np.random.default_rng(100 + fmt)
    idx = rng.choice(v.size, size=40_000, replace=False)
    for i in idx:
        x = float(v[i])
        assert orc.fp8_encode(x, fmt) == ref_encode(x, fmt), (fmt, x)


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_all_bf16_cast_points_match_independent(orc, fmt):
    """Every bf16 pattern through the element-wise cast (bf16 -> fp32 -> * scale)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for scale in (1.0, 3.5, 2.0 ** -20):
        out = orc.cast_points(bits, np.float32(scale), fmt)
        f = (bits.astype(np.uint32) << 16).view(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            p = (f * np.float32(scale)).astype(np.float32)
        for i in range(0, 65536, 7):
            if np.isnan(p[i]):
                assert is_nan_code(int(out[i]), fmt)
            else:
                x = float(p[i])
                exp = ref_encode(x if np.isfinite(p[i]) else math.copysign(1e300, x), fmt)
                assert out[i] == exp, (fmt, scale, hex(int(bits[i])), hex(int(out[i])), hex(exp))


def test_nan_and_inf_inputs(orc):
    for fmt in ALL_FMTS:
        assert is_nan_code(orc.fp8_encode(float("nan"), fmt), fmt)
        assert orc.fp8_encode(float("inf"), fmt) == orc.fp8_max_code(fmt)
        assert orc.fp8_encode(float("-inf"), fmt) == 0x80 | orc.fp8_max_code(fmt)
    assert orc.fp8_encode(-0.0, 0) == 0x80
    assert orc.fp8_encode(-0.0, 1) == 0x80
    assert orc.fp8_encode(-0.0, 2) == 0x00
    assert orc.fp8_encode(-0.0, 3) == 0x00
