"""GPU parity of fp8_blockwise_quantize against the oracle (bytes bit-exact
with NaN by class, every scale byte of the MX scale layout), and of the
block-scaled GEMM on blockwise operands (operands from the oracle's
quantize, tolerance |out - ref| <= 2e-3 * bound + 1e-5 + 2^-8 max(|ref|, |out|))."""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import assert_codes_equal, bits, check_gemm, mx_tiled, sample_points

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    fp8.load_library()


def gen_x(shape, seed, spread=8):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    if shape[0] > 0:
        x = x * torch.exp2(torch.randint(-spread, spread + 1, (shape[0], 1), generator=g).float())
    return x.to(torch.bfloat16)


def compare_bw(orc, x, fmt, block_rows, layouts=3, what="", xd=None):
    """xd: the device copy of x to quantize (default x.to(DEV)), e.g. a strided view"""
    ref = orc.blockwise_quantize(bits(x), fmt, block_rows, layouts)
    q = fp8.blockwise_quantize(x.to(DEV) if xd is None else xd, fmt, block_rows, layouts)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    rows = x.shape[0]
    if layouts & 1:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, f"{what} q_row")
        e = mx_tiled(ref["s_row"])
        assert np.array_equal(q.s_row.cpu().numpy()[:e.size], e), f"{what} s_row"
    if layouts & 2:
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :rows], ref["q_colT"], fmt, f"{what} q_colT")
        e = mx_tiled(ref["s_col"])
        assert np.array_equal(q.s_col.cpu().numpy()[:e.size], e), f"{what} s_col"
    return q, ref


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 1024)])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("block_rows", [1, 128])
def test_blockwise_quantize(orc, shape, fmt, block_rows):
    compare_bw(orc, gen_x(shape, seed=shape[0] + shape[1] + fmt + block_rows), fmt, block_rows,
               what=f"{shape} f{fmt} b{block_rows}")


@pytest.mark.parametrize("rows", [1, 37, 130, 253])
def test_blockwise_row_only_ragged_rows(orc, rows):
    compare_bw(orc, gen_x((rows, 256), seed=rows), 0, 1, layouts=1, what=f"rows {rows}")


@pytest.mark.parametrize("block_rows", [1, 128])
def test_blockwise_special_values(orc, block_rows):
    g = torch.Generator().manual_seed(3)
    x = synth.randomize_special(gen_x((256, 256), seed=5), g, frac=0.02)
    x[0:128, 0:128] = 0.0                       # an all-zero weight block / zero row blocks
    x[130, 7] = float("nan")
    x[140, 200] = float("inf")
    x[200, 0:128] = 2.0 ** -133                 # subnormal maxima
    compare_bw(orc, x, 1, block_rows, what=f"special b{block_rows}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_blockwise_every_bf16_pattern(orc, fmt):
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(2))
    for block_rows in (1, 128):
        compare_bw(orc, pats[perm].reshape(256, 256), fmt, block_rows, what=f"patterns f{fmt} b{block_rows}")


@pytest.mark.parametrize("block_rows", [1, 128])
def test_blockwise_many_tiles_per_block(orc, block_rows):
    """512 tiles of 128 x 128, more than the persistent grid holds: blocks
    convert one tile while the next one's loads are in flight."""
    compare_bw(orc, gen_x((4096, 2048), seed=11 + block_rows), 1, block_rows, what=f"4096x2048 b{block_rows}")


@pytest.mark.parametrize("block_rows", [1, 128])
def test_blockwise_rows_not_32_byte_aligned(orc, block_rows):
    """Row pitch cols + 8 (rows 16-byte but not 32-byte aligned): the 16-byte load path."""
    x = gen_x((384, 384), seed=21)
    pad = torch.zeros((384, 392), dtype=torch.bfloat16)
    pad[:, :384] = x
    compare_bw(orc, x, 0, block_rows, what=f"ld 392 b{block_rows}", xd=pad.to(DEV)[:, :384])


def test_blockwise_row_output_16_byte_aligned(orc):
    """q_row 16-byte but not 32-byte aligned: the row layout's 16-byte stores."""
    x = gen_x((256, 384), seed=23)
    ref = orc.blockwise_quantize(bits(x), 0, 1, 1)
    rows, cols = x.shape
    buf = torch.zeros(rows * cols + 48, dtype=torch.uint8, device=DEV)
    off = 16 if buf.data_ptr() % 32 == 0 else 0  # a 16-byte but not 32-byte aligned start
    q_row = buf[off:off + rows * cols]
    s_row = torch.zeros(fp8.fp8_mx_scale_bytes(rows, cols // 32), dtype=torch.uint8, device=DEV)
    xd = x.to(DEV)
    fp8.fp8_blockwise_quantize(xd, rows, cols, cols, 0, 1, 1, q_row, s_row, None, 0, None)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    assert_codes_equal(q_row.cpu().numpy().reshape(rows, cols), ref["q_row"], 0, "q_row at +16")
    e = mx_tiled(ref["s_row"])
    assert np.array_equal(s_row.cpu().numpy()[:e.size], e)
    assert (buf[:off].cpu().numpy() == 0).all() and (buf[off + rows * cols:].cpu().numpy() == 0).all()


@pytest.mark.parametrize("block_rows", [1, 128])
def test_blockwise_colT_pitch_16_not_32(orc, block_rows):
    """Transposed layout at a row pitch of rows + 16 (16-byte but not 32-byte
    aligned rows); the pitch's padding bytes stay untouched."""
    x = gen_x((256, 256), seed=41)
    ref = orc.blockwise_quantize(bits(x), 1, block_rows, 2)
    rows, cols = x.shape
    ld = rows + 16
    q_colT = torch.zeros((cols, ld), dtype=torch.uint8, device=DEV)
    s_col = torch.zeros(fp8.fp8_mx_scale_bytes(cols, rows // 32), dtype=torch.uint8, device=DEV)
    fp8.fp8_blockwise_quantize(x.to(DEV), rows, cols, cols, 1, block_rows, 2, None, None, q_colT, ld, s_col)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    got = q_colT.cpu().numpy()
    assert_codes_equal(got[:, :rows], ref["q_colT"], 1, f"q_colT pitch {ld} b{block_rows}")
    assert (got[:, rows:] == 0).all()
    e = mx_tiled(ref["s_col"])
    assert np.array_equal(s_col.cpu().numpy()[:e.size], e)


def test_blockwise_llama_weight_full(orc):
    """Llama-3-8B W_gate [14336, 4096], 128 x 128 blocks, both layouts, in full."""
    g = torch.Generator().manual_seed(1)
    w = (torch.randn((14336, 4096), generator=g) * 0.02).to(torch.bfloat16)
    compare_bw(orc, w, 0, 128, what="llama W_gate")


def up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("shape", [(128, 256, 128), (200, 384, 512), (384, 640, 1024)])
def test_blockwise_gemm_small(orc, shape):
    """Activation (1 x 128) x weight (128 x 128) through fp8_mx_gemm."""
    M, N, K = shape
    qa = orc.blockwise_quantize(bits(gen_x((M, K), seed=M)), 0, 1, layouts=1)
    Np = -(-N // 128) * 128
    qb = orc.blockwise_quantize(bits(gen_x((Np, K), seed=N)), 0, 128, layouts=1)
    B, sB = qb["q_row"][:N], qb["s_row"][:N]
    C = fp8.mx_gemm(up(qa["q_row"]), 0, up(mx_tiled(qa["s_row"])), up(B), 0, up(mx_tiled(sB)))
    assert fp8.fp8_sync_status() == 0
    ref, bound = orc.mx_gemm(qa["q_row"], 0, qa["s_row"], B, 0, sB)
    check_gemm(C.float().cpu().numpy(), ref, bound, f"blockwise {shape}")


def test_blockwise_gemm_llama_dgrad_sampled(orc):
    """dX = dY W on blockwise operands: dY [8192, 14336] E5M2 1 x 128 row
    layout, W [14336, 4096] E4M3 128 x 128 transposed layout; sampled."""
    M, N, K = 8192, 4096, 14336
    g = torch.Generator().manual_seed(7)
    dy = (torch.randn((M, K), generator=g) * 1e-4).to(torch.bfloat16)
    w = (torch.randn((K, N), generator=g) * 0.02).to(torch.bfloat16)
    qa = orc.blockwise_quantize(bits(dy), 1, 1, layouts=1)
    qb = orc.blockwise_quantize(bits(w), 0, 128, layouts=2)
    C = fp8.mx_gemm(up(qa["q_row"]), 1, up(mx_tiled(qa["s_row"])), up(qb["q_colT"]), 0, up(mx_tiled(qb["s_col"])))
    assert fp8.fp8_sync_status() == 0
    pm, pn = sample_points(torch.Generator().manual_seed(8), M, N, n_rows=8, n_cols=8, n_rand=2048)
    ref, bound = orc.mx_gemm(qa["q_row"], 1, qa["s_row"], qb["q_colT"], 0, qb["s_col"], points=(pm, pn))
    check_gemm(C.float().cpu().numpy()[pm, pn], ref, bound, "blockwise dgrad")
