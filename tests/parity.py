"""Helpers shared by the GPU parity tests: comparisons against the oracle."""
import numpy as np
import torch

import synth

TOL_REL = 2e-3   # |out - ref| <= TOL_REL * sum_k |a_k b_k| * |sa sb| + TOL_ABS (+ the bf16 cast, below)
TOL_ABS = 1e-5
BF16_HALF_ULP_REL = 2.0 ** -8   # round-to-nearest into bf16 moves a value by at most 2^-8 of itself


def nan_mask(codes: np.ndarray, fmt: int) -> np.ndarray:
    c = codes.astype(np.int32)
    if fmt in (2, 3):  # fnuz: the single NaN code
        return c == 0x80
    if fmt == 0:
        return (c & 0x7F) == 0x7F
    return (c & 0x7F) > 0x7C


def assert_codes_equal(gpu: np.ndarray, ref: np.ndarray, fmt: int, what: str = ""):
    """Bit-exact byte comparison; NaN outputs are compared by class."""
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    ng, nr = nan_mask(gpu, fmt), nan_mask(ref, fmt)
    bad = (ng != nr) | ((gpu != ref) & ~nr)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(f"{what}: {int(bad.sum())} byte mismatches, first at {idx.tolist()}: "
                             f"gpu {[hex(int(gpu[tuple(i)])) for i in idx]} ref {[hex(int(ref[tuple(i)])) for i in idx]}")


def assert_f32_bits_equal(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    g = np.ascontiguousarray(gpu, np.float32)
    r = np.ascontiguousarray(ref, np.float32)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    same = (g.view(np.uint32) == r.view(np.uint32)) | (np.isnan(g) & np.isnan(r))
    if not same.all():
        idx = np.argwhere(~same)[:8]
        raise AssertionError(f"{what}: {int((~same).sum())} fp32 mismatches at {idx.tolist()}: "
                             f"gpu {g[~same][:8]} ref {r[~same][:8]}")


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_gemm(out, ref, bound, what="", strict=False):
    """GEMM tolerance, elementwise:

        |out - ref| <= 2e-3 * bound + 1e-5            (the stated bound)
                       + 2^-8 * max(|ref|, |out|)     only where |ref| > bound / 16

    The last term is the bf16 output cast (half a bf16 ulp), which no bf16
    output can avoid where one product dominates a sum (|ref| close to bound,
    as with the tiny workload's 50x outliers: there half an ulp exceeds
    2e-3 * bound).  Where |ref| <= bound / 16 the cast moves a value by at most
    2^-12 * bound, which fits inside the stated bound together with the fp32
    accumulation error, so the stated bound alone applies.  strict=True asserts
    the stated bound on every element (random-sign data at large K, where
    |ref| / bound is about 1 / sqrt(K)).
    Returns the largest err / bound seen (the margin against 2e-3).
    """
    out = np.asarray(out, np.float64)
    err = np.abs(out - ref)
    lim = TOL_REL * bound + TOL_ABS
    if not strict:
        lim = lim + np.where(np.abs(ref) > bound / 16, BF16_HALF_ULP_REL * np.maximum(np.abs(ref), np.abs(out)), 0.0)
    bad = ~(err <= lim)
    if bad.any():
        i = np.argwhere(bad)[:6]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance{' (strict)' if strict else ''}; "
                             f"first {i.tolist()}: out {out[bad][:6]} ref {ref[bad][:6]} bound {bound[bad][:6]}")
    denom = np.where(bound > 0, bound, 1.0)
    return float((err / denom).max()) if err.size else 0.0


def finite_codes(gen: torch.Generator, shape, fmt: int) -> torch.Tensor:
    """Random FP8 codes with NaN / Inf codes replaced (CPU uint8)."""
    c = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32)
    if fmt == 0:
        bad = (c & 0x7F) == 0x7F
    else:
        bad = (c & 0x7F) >= 0x7C
    c[bad] = 0x30
    return c.to(torch.uint8)


def realistic_codes(gen: torch.Generator, shape, fmt: int) -> torch.Tensor:
    """Codes of N(0,1) values scaled so the max lands near the format max."""
    x = torch.randn(shape, generator=gen)
    s = (448.0 if fmt == 0 else 57344.0) / float(x.abs().max())
    dt = torch.float8_e4m3fn if fmt == 0 else torch.float8_e5m2
    return (x * s).to(dt).view(torch.uint8)


def sample_points(gen: torch.Generator, M: int, N: int, n_rows=64, n_cols=64, n_rand=4096):
    """64 full rows + 64 full columns + random points (numpy int64 pm, pn)."""
    rows = torch.randperm(M, generator=gen)[:min(n_rows, M)].numpy()
    cols = torch.randperm(N, generator=gen)[:min(n_cols, N)].numpy()
    pm = [np.repeat(rows, N), np.tile(np.arange(N), len(rows)).astype(np.int64)]
    pc = [np.tile(np.arange(M), len(cols)).astype(np.int64), np.repeat(cols, M)]
    rm = torch.randint(0, M, (n_rand,), generator=gen).numpy()
    rn = torch.randint(0, N, (n_rand,), generator=gen).numpy()
    return (np.concatenate([pm[0], pc[0], rm]).astype(np.int64),
            np.concatenate([pm[1], pc[1], rn]).astype(np.int64))


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def mx_tiled(plain: np.ndarray) -> np.ndarray:
    """Plain E8M0 codes [R][KB] -> the bytes of the MX scale layout: K tiles
    of four blocks, [ceil(KB/4)][roundup(R, 128)][4], each 128-row block of
    a K tile stored as [32 lanes][4 row groups][4 blocks] (row 32 j + L at
    lane L, word j); pad bytes 0."""
    R, KB = plain.shape
    KT = -(-KB // 4)
    Rs = -(-R // 128) * 128
    padded = np.zeros((Rs, KT * 4), np.uint8)
    padded[:R, :KB] = plain
    t = padded.reshape(Rs // 128, 4, 32, KT, 4)          # [row block][j][L][kt][block]
    return np.ascontiguousarray(t.transpose(3, 0, 2, 1, 4)).reshape(-1)