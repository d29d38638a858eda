"""GPU parity of the fused MoE prologues of the rowwise recipe
(fp8_permute_quantize, fp8_swiglu_quantize) against the oracle.

Gather: bytes bit-exact (NaN by class) and every fp32 row / (group, column)
scale_inv bit for bit against the oracle's quantize of the gathered rows.

SwiGLU: the kernel's h (the optional bf16 copy) within one bf16 ulp of the
oracle's exact h, element by element, and the bytes and scales bit-exact
against the oracle's quantize of the kernel's own h.

Both run the grouped rowwise passes of fp8_quantize with the prologue
applied to what each pass reads; the cases cover empty groups, a large group
next to runs of small ones, columns that are not a multiple of the tile
widths, one layout at a time, margins and the tensor amax."""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import assert_codes_equal, assert_f32_bits_equal, bits
from test_gpu_moe_fused import check_h, gen, h_bits, routing

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    fp8.load_library()


def check(q, ref, fmt, layouts, off, what, amax=None):
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    rows = int(off[-1])
    G = len(off) - 1
    if layouts & fp8.LAYOUT_ROW:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, f"{what} q_row")
        assert_f32_bits_equal(q.scale_inv_row.cpu().numpy()[:rows], ref["scale_inv_row"], f"{what} sinv_row")
    if layouts & fp8.LAYOUT_COLT:
        P = ref["q_colT"].shape[1]
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :P], ref["q_colT"], fmt, f"{what} q_colT")
        assert_f32_bits_equal(q.scale_inv_col.cpu().numpy().reshape(G, -1), ref["scale_inv_col"],
                              f"{what} sinv_col")
    if amax is not None:
        assert_f32_bits_equal(amax.cpu().numpy(), np.array([ref["amax"]], np.float32), f"{what} amax")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("fmt", [0, 1])
def test_permute_quantize_grouped(orc, fmt):
    src, off = routing(T=300, E=8, topk=3, seed=fmt, empty=(2, 5))
    x = gen((300, 160), seed=4 + fmt)
    ref = orc.permute_quantize(bits(x), src, fmt, orc.ROWWISE, off)
    amax = torch.full((1,), 5.0, device=DEV)
    q = fp8.permute_quantize(x.to(DEV), dev(src), fmt, dev(off), off, amax_out=amax)
    check(q, ref, fmt, 3, off, f"permute f{fmt}", amax)


@pytest.mark.parametrize("layouts", [1, 2])
def test_permute_quantize_single_layout_margin(orc, layouts):
    src, off = routing(T=200, E=16, topk=2, seed=7, empty=(0, 9, 15))
    x = gen((200, 1048), seed=8)
    ref = orc.permute_quantize(bits(x), src, 0, orc.ROWWISE, off, margin=2, layouts=layouts)
    q = fp8.permute_quantize(x.to(DEV), dev(src), 0, dev(off), off, layouts=layouts, margin=2)
    check(q, ref, 0, layouts, off, f"permute layouts {layouts}")


def test_permute_bad_index_reported(orc):
    x = gen((20, 64), seed=1)
    src = np.array([0, 1, 25, 3], np.int32)                          # 25 is outside x
    off = np.array([0, 3, 4], np.int32)
    q = fp8.permute_quantize(x.to(DEV), dev(src), 0, dev(off), off, layouts=fp8.LAYOUT_ROW)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 1                                # FP8_ERR_INVALID_ARG
    assert (q.q_row[2] == 0).all()                                   # read as a zero row
    assert fp8.fp8_sync_status() == 0


def test_permute_large_group_and_ragged_columns(orc):
    """cols = 4104 (a multiple of 8 only), a 5000-row group next to runs of
    small and empty groups; two calls give the same bytes."""
    sizes = np.array([5, 0, 17, 5000, 1, 0, 0, 33, 700, 2, 0, 64, 2500, 9], np.int64)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(off[-1])
    x = gen((3000, 4104), seed=21)
    src = np.random.default_rng(5).integers(0, 3000, size=M).astype(np.int32)
    ref = orc.permute_quantize(bits(x), src, 1, orc.ROWWISE, off)
    q = fp8.permute_quantize(x.to(DEV), dev(src), 1, dev(off), off)
    check(q, ref, 1, 3, off, "large group")
    q2 = fp8.permute_quantize(x.to(DEV), dev(src), 1, dev(off), off)
    torch.cuda.synchronize()
    assert torch.equal(q.q_row, q2.q_row) and torch.equal(q.q_colT, q2.q_colT)


def swiglu_case(orc, gu, fmt, layouts, off, what, margin=0):
    rows, F2 = gu.shape
    F = F2 // 2
    h = torch.empty((rows, F), dtype=torch.bfloat16, device=DEV)
    amax = torch.zeros(1, device=DEV)
    q = fp8.swiglu_quantize(gu.to(DEV), fmt, dev(off), off, layouts=layouts, h_out=h, margin=margin, amax_out=amax)
    torch.cuda.synchronize()
    hg = h_bits(h)
    gb = bits(gu)
    check_h(hg, orc.swiglu_bf16(gb[:, :F], gb[:, F:]), what)
    ref = orc.quantize(hg, fmt, orc.ROWWISE, margin=margin, layouts=layouts, offsets=off)
    check(q, ref, fmt, layouts, off, what, amax)
    return q, hg


@pytest.mark.parametrize("fmt", [0, 1])
def test_swiglu_quantize_grouped(orc, fmt):
    sizes = [10, 0, 97, 1, 0, 116]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows, F = int(off[-1]), 200
    gu = gen((rows, 2 * F), seed=20 + fmt, scale=3.0)
    g = torch.Generator().manual_seed(5)
    gu = synth.randomize_special(gu, g, frac=0.01)
    gu[3, 7] = 120.0
    gu[4, 9] = -120.0
    gu[5, 11] = -float("inf")
    swiglu_case(orc, gu, fmt, 3, off, f"swiglu rowwise f{fmt}")


@pytest.mark.parametrize("layouts", [1, 2])
def test_swiglu_quantize_single_layout_without_h(orc, layouts):
    off = np.array([0, 40, 40, 130], np.int32)
    gu = gen((130, 2 * 264), seed=31)
    _, hg = swiglu_case(orc, gu, 1, layouts, off, f"swiglu layouts {layouts}", margin=1)
    q = fp8.swiglu_quantize(gu.to(DEV), 1, dev(off), off, layouts=layouts, margin=1)
    ref = orc.quantize(hg, 1, orc.ROWWISE, margin=1, layouts=layouts, offsets=off)
    check(q, ref, 1, layouts, off, f"swiglu layouts {layouts}, no h")


def test_dsv3_shapes(orc):
    """DeepSeek-V3 shapes: 2048 tokens x top-8 of 256 experts (8 empty),
    hidden 7168; SwiGLU of the [16384, 2 x 2048] gate|up output."""
    src, off = routing(T=2048, E=256, topk=8, seed=3, empty=tuple(range(0, 256, 32)))
    x = gen((2048, 7168), seed=41)
    ref = orc.permute_quantize(bits(x), src, 0, orc.ROWWISE, off)
    q = fp8.permute_quantize(x.to(DEV), dev(src), 0, dev(off), off)
    check(q, ref, 0, 3, off, "dsv3 permute")
    gu = gen((16384, 4096), seed=42, scale=2.0)
    swiglu_case(orc, gu, 0, 3, off, "dsv3 swiglu")
