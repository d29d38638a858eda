"""GPU parity of the fused MoE prologues (fp8_mx_permute_quantize,
fp8_mx_swiglu_quantize) against the oracle.

Gather: element bytes bit-exact (NaN by class) and every E8M0 scale byte
against the oracle's gather + MX quantize.

SwiGLU: the oracle's h is the exact bf16_rne(silu(g) * u); the kernel
evaluates silu in fp32 with the fast exponential, so its h (the optional bf16
copy) is checked within one bf16 ulp of the oracle's, element by element
(the number of elements that differ is reported), and its bytes and scales
bit-exact against the oracle's MX quantize of the kernel's own h."""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import assert_codes_equal, bits, mx_tiled

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    fp8.load_library()


def routing(T, E, topk, seed, empty=()):
    """Each token to `topk` distinct experts (none of `empty`); returns the
    source row of every routed row in expert order and the group offsets."""
    g = np.random.default_rng(seed)
    allowed = np.array([e for e in range(E) if e not in empty])
    experts = np.stack([g.choice(allowed, size=topk, replace=False) for _ in range(T)])
    tok = np.repeat(np.arange(T), topk)
    exp = experts.reshape(-1)
    order = np.argsort(exp, kind="stable")
    src = tok[order].astype(np.int32)
    sizes = np.bincount(exp, minlength=E)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return src, off


def gen(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    x = x * torch.exp2(torch.randint(-4, 5, (shape[0], 1), generator=g).float())
    return x.to(torch.bfloat16)


def check(q, ref, fmt, layouts, what):
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    P = q.scale_rows
    if layouts & fp8.LAYOUT_ROW:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, f"{what} q_row")
        e = mx_tiled(ref["s_row"])
        assert np.array_equal(q.s_row.cpu().numpy()[:e.size], e), f"{what} s_row"
    if layouts & fp8.LAYOUT_COLT:
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :P], ref["q_colT"], fmt, f"{what} q_colT")
        e = mx_tiled(ref["s_col"])
        assert np.array_equal(q.s_col.cpu().numpy()[:e.size], e), f"{what} s_col"


@pytest.mark.parametrize("fmt", [0, 1])
def test_permute_quantize_grouped(orc, fmt):
    src, off = routing(T=300, E=8, topk=3, seed=fmt, empty=(2, 5))
    x = gen((300, 160), seed=4 + fmt)
    ref = orc.mx_permute_quantize(bits(x), src, fmt, 3, offsets=off, align=128)
    q = fp8.mx_permute_quantize(x.to(DEV), torch.from_numpy(src).to(DEV), fmt, 3,
                                group_offsets=torch.from_numpy(off).to(DEV), host_offsets=torch.from_numpy(off))
    check(q, ref, fmt, 3, f"permute grouped f{fmt}")


def test_permute_quantize_ungrouped_and_repeats(orc):
    g = np.random.default_rng(9)
    src = g.integers(0, 50, size=128).astype(np.int32)
    src[:8] = 7                                      # one token many times
    x = gen((50, 96), seed=11)
    ref = orc.mx_permute_quantize(bits(x), src, 0, 3)
    q = fp8.mx_permute_quantize(x.to(DEV), torch.from_numpy(src).to(DEV), 0, 3)
    check(q, ref, 0, 3, "permute ungrouped")


def test_permute_bad_index_reported():
    x = gen((20, 64), seed=1).to(DEV)
    src = torch.tensor([0, 1, 25, 3], dtype=torch.int32, device=DEV)   # 25 is outside
    q = fp8.mx_permute_quantize(x, src, 0, fp8.LAYOUT_ROW)
    assert fp8.fp8_sync_status() == 1                                   # FP8_ERR_INVALID_ARG
    assert (q.q_row[2] == 0).all()                                      # read as a zero row
    assert fp8.fp8_sync_status() == 0


def ordered(bits16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers in the order of their values (-0 and +0
    both 0), so adjacent representable values differ by one."""
    b = bits16.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def check_h(h_gpu: np.ndarray, h_ref: np.ndarray, what: str) -> int:
    """Within one bf16 ulp of the oracle's h (NaN by class); returns how many
    elements differ."""
    nan_g = (h_gpu & 0x7FFF) > 0x7F80
    nan_r = (h_ref & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    d = np.abs(ordered(h_gpu[~nan_g]) - ordered(h_ref[~nan_r]))
    assert d.size == 0 or d.max() <= 1, f"{what}: {int((d > 1).sum())} elements more than one bf16 ulp off"
    n = int((d != 0).sum())
    print(f"{what}: {n} of {d.size} elements of h one bf16 ulp from the oracle's, the rest equal")
    return n


def h_bits(h: torch.Tensor) -> np.ndarray:
    return h.cpu().view(torch.int16).numpy().view(np.uint16)


def swiglu_case(orc, gu, fmt, layouts, off, what):
    rows, F2 = gu.shape
    F = F2 // 2
    h = torch.empty((rows, F), dtype=torch.bfloat16, device=DEV)
    q = fp8.mx_swiglu_quantize(gu.to(DEV), fmt, layouts, h_out=h,
                               group_offsets=None if off is None else torch.from_numpy(off).to(DEV),
                               host_offsets=None if off is None else torch.from_numpy(off))
    torch.cuda.synchronize()
    hg = h_bits(h)
    gb = bits(gu)
    check_h(hg, orc.swiglu_bf16(gb[:, :F], gb[:, F:]), what)
    ref = orc.mx_quantize(hg, fmt, layouts, offsets=off, align=128)
    check(q, ref, fmt, layouts, what)
    return q, hg


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("grouped", [False, True])
def test_swiglu_quantize(orc, fmt, grouped):
    rows, F = (224, 192) if grouped else (128, 160)
    gu = gen((rows, 2 * F), seed=20 + fmt, scale=3.0)
    g = torch.Generator().manual_seed(5)
    gu = synth.randomize_special(gu, g, frac=0.01)
    gu[3, 7] = 120.0                                 # e^-g far below an ulp of 1: silu(g) = g
    gu[4, 9] = -120.0                                # silu(g) * u below the smallest bf16
    gu[5, 11] = -float("inf")                        # silu(-Inf) = -0
    off = None
    if grouped:
        sizes = [10, 0, 97, 1, 0, 116]
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    swiglu_case(orc, gu, fmt, 3, off, f"swiglu f{fmt} g{grouped}")


@pytest.mark.parametrize("u", [1.0, -0.75, 3.0e4, -1e-5, 2.0 ** 40])
def test_swiglu_every_gate_value(orc, u):
    """Every bf16 pattern as the gate (NaN and +-Inf included), with one up
    value per case, row layout."""
    gate = torch.arange(0, 0x10000, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(64, 1024)
    gu = torch.cat([gate, torch.full((64, 1024), u, dtype=torch.bfloat16)], dim=1)
    swiglu_case(orc, gu, 0, fp8.LAYOUT_ROW, None, f"every gate, u = {u}")


def test_swiglu_without_h_and_row_only(orc):
    """Without the bf16 copy: the bytes equal those of a call that writes
    it, and so the oracle's MX quantize of that h."""
    gu = gen((40, 128), seed=31)
    _, hg = swiglu_case(orc, gu, 0, fp8.LAYOUT_ROW, None, "swiglu row only, with h")
    q = fp8.mx_swiglu_quantize(gu.to(DEV), 0, fp8.LAYOUT_ROW)
    check(q, orc.mx_quantize(hg, 0, fp8.LAYOUT_ROW), 0, fp8.LAYOUT_ROW, "swiglu row only")


def test_dsv3_routed_tokens_and_swiglu(orc):
    """DeepSeek-V3 shapes: 2048 tokens x top-8 of 256 experts (8 empty),
    hidden 7168; SwiGLU of the [16384, 2 x 2048] gate|up output."""
    src, off = routing(T=2048, E=256, topk=8, seed=3, empty=tuple(range(0, 256, 32)))
    x = gen((2048, 7168), seed=41)
    ref = orc.mx_permute_quantize(bits(x), src, 0, 3, offsets=off, align=128)
    q = fp8.mx_permute_quantize(x.to(DEV), torch.from_numpy(src).to(DEV), 0, 3,
                                group_offsets=torch.from_numpy(off).to(DEV), host_offsets=torch.from_numpy(off))
    check(q, ref, 0, 3, "dsv3 permute")
    gu = gen((16384, 4096), seed=42, scale=2.0)
    swiglu_case(orc, gu, 0, 3, off, "dsv3 swiglu")
