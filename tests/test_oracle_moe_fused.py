"""Pins of the oracle's MoE prologues (CPU only): the gather that permutes
token rows into expert order and SwiGLU, fused in front of the MX quantize
("FP8 Training on AMD GPUs with TorchTitan and TorchAO": a five-kernel eager
chain replaced by one fused kernel on the MoE path).

  * exp_f32 (the fixed fp32 exp of the SwiGLU definition) against the
    mathematical exp within its stated error, plus its special cases;
  * bf16_rne against PyTorch's fp32 -> bf16 conversion (library RNE);
  * SwiGLU against the double-precision silu(g) * u: exact after bf16
    rounding except where the fp32 evaluation sits next to a rounding
    boundary (then one bf16 ulp), and the limits silu(+large) = g,
    silu(-large) = -0;
  * the gather: identity = plain quantize, a permutation permutes the row
    layout, repeated indices repeat rows.
"""
import math

import numpy as np
import pytest
import torch

from test_oracle_mx import bf16_bits, bits_to_f64


def test_exp_f32_accuracy_and_specials(orc):
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), np.linspace(-1, 1, 2001)]).astype(np.float32)
    worst = 0.0
    prev = -1.0
    for x in np.sort(xs):
        e = float(orc.exp_f32(float(x)))
        ref = math.exp(float(x))
        rel = abs(e - ref) / ref
        worst = max(worst, rel)
        assert e >= prev                       # monotone on the sorted sweep
        prev = e
    assert worst < 4 * 2.0 ** -23, worst       # a few fp32 ulps
    assert orc.exp_f32(0.0) == 1.0
    assert math.isnan(orc.exp_f32(float("nan")))
    assert orc.exp_f32(89.0) == float("inf")
    assert orc.exp_f32(-105.0) == 0.0


def test_bf16_rne_matches_torch(orc):
    g = np.random.default_rng(0)
    u = g.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    u[:2000] = (u[:2000] & 0xFFFF0000) | 0x8000        # exact ties
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_rne(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)


def _silu_exact(g, u):
    return (g / (1.0 + np.exp(-g))) * u


def test_swiglu_against_double(orc):
    g = np.random.default_rng(1)
    gv = (g.standard_normal(200000) * 4).astype(np.float32)
    uv = (g.standard_normal(200000) * 2).astype(np.float32)
    gb, ub = bf16_bits(gv), bf16_bits(uv)
    h = orc.swiglu_bf16(gb, ub)
    hv = bits_to_f64(h)
    with np.errstate(over="ignore"):
        exact = _silu_exact(bits_to_f64(gb), bits_to_f64(ub))
    exact_bf16 = bits_to_f64(bf16_bits(exact.astype(np.float32)))
    same = hv == exact_bf16
    assert same.mean() > 0.999
    # elsewhere within one bf16 ulp of the exact value
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-38))) - 7)
    assert np.all(np.abs(hv - exact) <= ulp + 1e-300)


def test_swiglu_limits(orc):
    g = bf16_bits(np.array([0.0, 100.0, -100.0, 300.0, -300.0, float("nan"), 1.0], np.float32))
    u = bf16_bits(np.array([3.0, 1.5, 2.0, -1.0, -2.0, 1.0, float("nan")], np.float32))
    h = bits_to_f64(orc.swiglu_bf16(g, u))
    assert h[0] == 0.0
    assert h[1] == 150.0                      # exp(-100) = 0: silu(g) = g
    assert h[2] == 0.0 and np.signbit(h[2])   # exp(100) = Inf: silu(g) = -0; -0 * 2 = -0
    assert h[3] == -300.0
    assert h[4] == 0.0 and not np.signbit(h[4])   # -0 * -2 = +0
    assert np.isnan(h[5]) and np.isnan(h[6])


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
