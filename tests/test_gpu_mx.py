"""GPU parity of the MXFP8 path (fp8_mx_quantize, fp8_mx_gemm,
fp8_mx_grouped_gemm) against the oracle.

Quantize: bit-exact element bytes (NaN compared by class) and E8M0 scale
bytes over the whole scale buffers (pad bytes included), for both layouts,
ragged shapes, special values, every bf16 pattern, grouped tensors with
empty groups and a full-size Llama-3-8B activation.

GEMM: operands are produced by the oracle's MX quantize of seeded inputs
(never by the GPU), uploaded in the MX scale layout, and the bf16 result is
compared with the oracle's fp64 block-scaled product under the GEMM
tolerance |out - ref| <= 2e-3 * bound + 1e-5 + 2^-8 * max(|ref|, |out|).
"""
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


def gen_x(shape, seed, scale=1.0, spread=6):
    """bf16 values N(0, 1) times a per-row power-of-two spread (exercises
    many block scales)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    if shape[0] > 0:
        x = x * torch.exp2(torch.randint(-spread, spread + 1, (shape[0], 1), generator=g).float())
    return x.to(torch.bfloat16)


def compare_mx(orc, x, fmt, layouts=3, offsets=None, what=""):
    xb = bits(x)
    ref = orc.mx_quantize(xb, fmt, layouts, offsets=offsets, align=fp8.MX_GROUP_ALIGN)
    dev_off = None if offsets is None else torch.as_tensor(np.asarray(offsets, np.int32), device=DEV)
    q = fp8.mx_quantize(x.to(DEV), fmt, layouts, group_offsets=dev_off,
                        host_offsets=None if offsets is None else torch.as_tensor(np.asarray(offsets, np.int32)))
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    P = q.scale_rows
    if layouts & fp8.LAYOUT_ROW:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, f"{what} q_row")
        exp = mx_tiled(ref["s_row"])
        got = q.s_row.cpu().numpy()
        assert got.size >= exp.size and np.array_equal(got[:exp.size], exp), f"{what} s_row"
    if layouts & fp8.LAYOUT_COLT:
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :P], ref["q_colT"], fmt, f"{what} q_colT")
        exp = mx_tiled(ref["s_col"])
        got = q.s_col.cpu().numpy()
        assert got.size >= exp.size and np.array_equal(got[:exp.size], exp), f"{what} s_col"
    return q, ref


# --- quantize ----------------------------------------------------------------

SHAPES = [(64, 128), (96, 160), (32, 32), (128, 4096), (320, 544), (1024, 96)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_quantize_both_layouts(orc, shape, fmt):
    compare_mx(orc, gen_x(shape, seed=shape[0] + shape[1] + fmt), fmt, 3, what=f"{shape} f{fmt}")


@pytest.mark.parametrize("rows", [1, 37, 62, 65, 130])
def test_mx_quantize_row_only_ragged_rows(orc, rows):
    """Row layout alone allows any row count; the scale rows are padded to 4."""
    compare_mx(orc, gen_x((rows, 224), seed=rows), 0, fp8.LAYOUT_ROW, what=f"rows {rows}")


@pytest.mark.parametrize("layouts", [1, 2])
def test_mx_quantize_single_layout(orc, layouts):
    compare_mx(orc, gen_x((192, 384), seed=3), 1, layouts, what=f"layouts {layouts}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_quantize_special_values(orc, fmt):
    g = torch.Generator().manual_seed(8 + fmt)
    x = synth.randomize_special(gen_x((128, 256), seed=10), g, frac=0.02)
    x[3, 5] = float("nan")
    x[40, 70] = float("inf")
    x[64:96, 128:160] = 0.0                 # all-zero blocks in both directions
    x[100, 200:232] = 1e38                  # huge block
    x[101, 0:32] = 2.0 ** -133              # bf16 subnormals
    compare_mx(orc, x, fmt, 3, what=f"special f{fmt}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_every_bf16_pattern(orc, fmt):
    """All 65536 bf16 patterns, laid out so each row block and each column
    block mixes magnitudes."""
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(1))
    compare_mx(orc, pats[perm].reshape(256, 256), fmt, 3, what=f"patterns f{fmt}")
    compare_mx(orc, pats.reshape(512, 128), fmt, 3, what=f"patterns sorted f{fmt}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_quantize_grouped(orc, fmt):
    sizes = [5, 0, 70, 1, 0, 129, 32, 300]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = gen_x((int(off[-1]), 160), seed=12 + fmt)
    q, _ = compare_mx(orc, x, fmt, 3, offsets=off, what=f"grouped f{fmt}")
    assert q.scale_rows == sum(-(-m // 128) * 128 for m in sizes)


def test_mx_quantize_grouped_row_only_and_all_empty(orc):
    sizes = [0, 3, 0]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    compare_mx(orc, gen_x((3, 64), seed=2), 0, fp8.LAYOUT_ROW, offsets=off, what="tiny grouped")
    off0 = np.zeros(4, np.int32)
    x = torch.zeros((0, 64), dtype=torch.bfloat16)
    q = fp8.mx_quantize(x.to(DEV), 1, 3, group_offsets=torch.as_tensor(off0, device=DEV),
                        host_offsets=torch.as_tensor(off0))
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0 and q.scale_rows == 0


def test_mx_quantize_bad_offsets_flagged():
    x = gen_x((64, 64), seed=1).to(DEV)
    off = torch.tensor([0, 40, 30, 64], dtype=torch.int32)      # decreasing
    q_row = torch.empty((64, 64), dtype=torch.uint8, device=DEV)
    s_row = torch.full((fp8.fp8_mx_scale_bytes(512, 2),), 7, dtype=torch.uint8, device=DEV)
    fp8.fp8_mx_quantize(x, 64, 64, 64, 0, fp8.LAYOUT_ROW, q_row, s_row, None, 0, None, off.to(DEV), 3)
    assert fp8.fp8_sync_status() == 1                            # FP8_ERR_INVALID_ARG
    assert (s_row.cpu() == 7).all()                             # nothing written
    assert fp8.fp8_sync_status() == 0


def test_mx_quantize_tall_band_walk(orc):
    """A tall tensor (65600 rows: tiles walked in bands of eight column tiles)
    with nine column tiles (a last band one tile wide) and a padding row tile
    past the data (rows rounded up to 128), both layouts in full."""
    compare_mx(orc, gen_x((65600, 1152), seed=43), 1, 3, what="65600x1152")


def test_mx_quantize_band_threshold_ragged_cols(orc):
    """Exactly the row count from which tiles are walked in column bands
    (65536), with ten column tiles the last of which is a quarter full."""
    compare_mx(orc, gen_x((65536, 1184), seed=47), 0, 3, what="65536x1184")


def test_mx_quantize_llama_activation_full(orc):
    """Llama-3-8B MLP input [8192, 4096], both layouts, compared in full."""
    g = torch.Generator().manual_seed(1)
    x = torch.randn((8192, 4096), generator=g).to(torch.bfloat16)
    compare_mx(orc, x, 0, 3, what="llama X")


def test_mx_quantize_row_output_16_byte_aligned(orc):
    """q_row 16-byte but not 32-byte aligned: the row layout's 16-byte stores."""
    x = gen_x((96, 160), seed=31)
    ref = orc.mx_quantize(bits(x), 1, fp8.LAYOUT_ROW, offsets=None, align=fp8.MX_GROUP_ALIGN)
    rows, cols = x.shape
    buf = torch.zeros(rows * cols + 48, dtype=torch.uint8, device=DEV)
    off = 16 if buf.data_ptr() % 32 == 0 else 0  # a 16-byte but not 32-byte aligned start
    q_row = buf[off:off + rows * cols]
    s_row = torch.zeros(fp8.fp8_mx_scale_bytes(rows, cols // 32), dtype=torch.uint8, device=DEV)
    fp8.fp8_mx_quantize(x.to(DEV), rows, cols, cols, 1, fp8.LAYOUT_ROW, q_row, s_row, None, 0, None)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    assert_codes_equal(q_row.cpu().numpy().reshape(rows, cols), ref["q_row"], 1, "q_row at +16")
    exp = mx_tiled(ref["s_row"])
    assert np.array_equal(s_row.cpu().numpy()[:exp.size], exp)
    assert (buf[:off].cpu().numpy() == 0).all() and (buf[off + rows * cols:].cpu().numpy() == 0).all()


def test_mx_quantize_colT_pitch_16_not_32(orc):
    """Transposed layout at a row pitch of rows + 16 (16-byte but not 32-byte
    aligned rows); the pitch's padding bytes stay untouched."""
    x = gen_x((64, 160), seed=37)
    ref = orc.mx_quantize(bits(x), 0, fp8.LAYOUT_COLT, offsets=None, align=fp8.MX_GROUP_ALIGN)
    rows, cols = x.shape
    ld = rows + 16
    q_colT = torch.zeros((cols, ld), dtype=torch.uint8, device=DEV)
    s_col = torch.zeros(fp8.fp8_mx_scale_bytes(cols, rows // 32), dtype=torch.uint8, device=DEV)
    fp8.fp8_mx_quantize(x.to(DEV), rows, cols, cols, 0, fp8.LAYOUT_COLT, None, None, q_colT, ld, s_col)
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    got = q_colT.cpu().numpy()
    assert_codes_equal(got[:, :rows], ref["q_colT"], 0, "q_colT pitch 80")
    assert (got[:, rows:] == 0).all()
    exp = mx_tiled(ref["s_col"])
    assert np.array_equal(s_col.cpu().numpy()[:exp.size], exp)


def test_mx_quantize_deterministic():
    x = gen_x((256, 512), seed=5).to(DEV)
    a = fp8.mx_quantize(x, 0)
    b = fp8.mx_quantize(x, 0)
    torch.cuda.synchronize()
    assert torch.equal(a.q_row, b.q_row) and torch.equal(a.s_row, b.s_row)
    assert torch.equal(a.q_colT[:, :256], b.q_colT[:, :256]) and torch.equal(a.s_col, b.s_col)


# --- GEMM --------------------------------------------------------------------

def mx_operand(orc, rows, K, fmt, seed, spread=4):
    ref = orc.mx_quantize(bits(gen_x((rows, K), seed, spread=spread)), fmt, fp8.LAYOUT_ROW)
    return ref["q_row"], ref["s_row"]


def up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


MX_SMALL = [(128, 224, 128), (1, 1, 32), (100, 40, 64), (130, 300, 160), (256, 448, 512), (300, 520, 1056),
            (129, 257, 4096), (257, 1, 32), (520, 264, 96)]


@pytest.mark.parametrize("shape", MX_SMALL)
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
def test_mx_gemm_small_full(orc, shape, fa, fb):
    M, N, K = shape
    A, sA = mx_operand(orc, M, K, fa, seed=M + K + fa)
    B, sB = mx_operand(orc, N, K, fb, seed=N + 2 * K + fb)
    C = fp8.mx_gemm(up(A), fa, up(mx_tiled(sA)), up(B), fb, up(mx_tiled(sB)))
    assert fp8.fp8_sync_status() == 0
    ref, bound = orc.mx_gemm(A, fa, sA, B, fb, sB)
    check_gemm(C.float().cpu().numpy(), ref, bound, f"mx {shape} {fa}{fb}")


def test_mx_gemm_wide_scale_spread(orc):
    """Block scales spread over 2^-40 .. 2^40 between rows and K blocks."""
    M, N, K = 256, 448, 1024
    A, sA = mx_operand(orc, M, K, 0, seed=1, spread=20)
    B, sB = mx_operand(orc, N, K, 0, seed=2, spread=20)
    C = fp8.mx_gemm(up(A), 0, up(mx_tiled(sA)), up(B), 0, up(mx_tiled(sB)))
    assert fp8.fp8_sync_status() == 0
    ref, bound = orc.mx_gemm(A, 0, sA, B, 0, sB)
    check_gemm(C.float().cpu().numpy(), ref, bound, "spread")


def test_mx_gemm_padded_ld_and_deterministic(orc):
    M, N, K = 200, 300, 256
    A, sA = mx_operand(orc, M, K, 0, seed=3)
    B, sB = mx_operand(orc, N, K, 1, seed=4)
    Ap = np.zeros((M, K + 64), np.uint8)
    Ap[:, :K] = A
    Cp = torch.zeros((M, N + 5), dtype=torch.bfloat16, device=DEV)
    fp8.mx_gemm(up(Ap), 0, up(mx_tiled(sA)), up(B), 1, up(mx_tiled(sB)), K=K, out=Cp[:, :N])
    C2 = fp8.mx_gemm(up(A), 0, up(mx_tiled(sA)), up(B), 1, up(mx_tiled(sB)))
    assert fp8.fp8_sync_status() == 0
    ref, bound = orc.mx_gemm(A, 0, sA, B, 1, sB)
    check_gemm(Cp[:, :N].float().cpu().numpy(), ref, bound, "padded ld")
    assert torch.equal(Cp[:, :N], C2)
    assert (Cp[:, N:] == 0).all()


def test_mx_gemm_llama_gate_sampled(orc):
    """Llama-3-8B gate projection fprop, M=8192 N=14336 K=4096, sampled."""
    M, N, K = 8192, 14336, 4096
    A, sA = mx_operand(orc, M, K, 0, seed=21, spread=1)
    B, sB = mx_operand(orc, N, K, 0, seed=22, spread=1)
    C = fp8.mx_gemm(up(A), 0, up(mx_tiled(sA)), up(B), 0, up(mx_tiled(sB)))
    assert fp8.fp8_sync_status() == 0
    g = torch.Generator().manual_seed(5)
    pm, pn = sample_points(g, M, N, n_rows=16, n_cols=16, n_rand=4096)
    ref, bound = orc.mx_gemm(A, 0, sA, B, 0, sB, points=(pm, pn))
    check_gemm(C.float().cpu().numpy()[pm, pn], ref, bound, "llama gate", strict=True)


# --- grouped GEMM ------------------------------------------------------------

def test_mx_grouped_m_small(orc):
    sizes = [5, 0, 200, 1, 0, 129, 64]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt, N, K = int(off[-1]), 384, 256     # N % 128 == 0: each expert's scale rows start a 128-row block
    xa = gen_x((Mt, K), seed=31)
    qa = orc.mx_quantize(bits(xa), 0, fp8.LAYOUT_ROW, offsets=off, align=128)
    B, sB = mx_operand(orc, G * N, K, 0, seed=32)
    C = fp8.mx_grouped_gemm(fp8.GROUPED_M, up(qa["q_row"]), 0, up(mx_tiled(qa["s_row"])), up(B), 0,
                            up(mx_tiled(sB)), up(off), Mt, N, K)
    assert fp8.fp8_sync_status() == 0
    poff = orc.padded_offsets_align(off, 128)
    out = C.float().cpu().numpy()
    for e in range(G):
        if sizes[e] == 0:
            continue
        r0, r1 = off[e], off[e + 1]
        ref, bound = orc.mx_gemm(qa["q_row"][r0:r1], 0, qa["s_row"][poff[e]:poff[e] + sizes[e]],
                                 B[e * N:(e + 1) * N], 0, sB[e * N:(e + 1) * N])
        check_gemm(out[r0:r1], ref, bound, f"mgroup e{e}")


def _mx_grouped_m_check(orc, sizes, N, K, seed, every=1):
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt = int(off[-1])
    xa = gen_x((Mt, K), seed=seed)
    qa = orc.mx_quantize(bits(xa), 0, fp8.LAYOUT_ROW, offsets=off, align=128)
    B, sB = mx_operand(orc, G * N, K, 0, seed=seed + 1)
    C = fp8.mx_grouped_gemm(fp8.GROUPED_M, up(qa["q_row"]), 0, up(mx_tiled(qa["s_row"])), up(B), 0,
                            up(mx_tiled(sB)), up(off), Mt, N, K)
    assert fp8.fp8_sync_status() == 0
    poff = orc.padded_offsets_align(off, 128)
    out = C.float().cpu().numpy()
    live = [e for e in range(G) if sizes[e] > 0]
    for e in live[::every] + live[-1:]:
        r0, r1 = off[e], off[e + 1]
        ref, bound = orc.mx_gemm(qa["q_row"][r0:r1], 0, qa["s_row"][poff[e]:poff[e] + sizes[e]],
                                 B[e * N:(e + 1) * N], 0, sB[e * N:(e + 1) * N])
        check_gemm(out[r0:r1], ref, bound, f"mgroup G{G} e{e}")


def test_mx_grouped_m_deep_k(orc):
    """Ten k-blocks per tile: the (four-stage) ring wraps inside every tile
    and across a CTA's tiles."""
    _mx_grouped_m_check(orc, [300, 0, 129, 64, 1, 256], 256, 1280, seed=61)


def test_mx_grouped_m_1000_groups(orc):
    """1000 groups: their tables leave no room for a fourth ring stage, so
    the M-grouped kernel runs its three-stage form (every 25th non-empty
    group and the last one checked in full)."""
    g = np.random.default_rng(63)
    sizes = [int(v) for v in g.integers(0, 5, size=1000)]
    _mx_grouped_m_check(orc, sizes, 128, 384, seed=63, every=25)


@pytest.mark.parametrize("NK", [(200, 300), (192, 296), (96, 520)])
def test_mx_grouped_k_small(orc, NK):
    """(200, 300) takes the direct-store epilogue; N % 32 == 0 with K % 8 == 0
    the TMA-store epilogue (partial tiles, K ending inside a box)."""
    sizes = [5, 0, 200, 1, 0, 129, 64]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt, (N, K) = int(off[-1]), NK
    qd = orc.mx_quantize(bits(gen_x((Mt, N), seed=41)), 1, fp8.LAYOUT_COLT, offsets=off, align=128)
    qx = orc.mx_quantize(bits(gen_x((Mt, K), seed=42)), 0, fp8.LAYOUT_COLT, offsets=off, align=128)
    P = qd["q_colT"].shape[1]
    # a NaN sentinel in every element: the empty groups' zeros are written, not left over
    sentinel = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = fp8.mx_grouped_gemm(fp8.GROUPED_K, up(qd["q_colT"]), 1, up(mx_tiled(qd["s_col"])), up(qx["q_colT"]), 0,
                            up(mx_tiled(qx["s_col"])), up(off), Mt, N, K, ld_T=P, out=sentinel)
    assert fp8.fp8_sync_status() == 0
    poff = orc.padded_offsets_align(off, 128)
    out = C.float().cpu().numpy()
    for e in range(G):
        if sizes[e] == 0:
            assert (out[e] == 0).all()
            continue
        a, b = int(poff[e]), int(poff[e + 1])
        ref, bound = orc.mx_gemm(qd["q_colT"][:, a:b], 1, qd["s_col"][:, a // 32:b // 32],
                                 qx["q_colT"][:, a:b], 0, qx["s_col"][:, a // 32:b // 32])
        check_gemm(out[e], ref, bound, f"kgroup e{e}")


def test_mx_grouped_k_many_tiles_per_cta(orc):
    """300 small groups with runs of empty ones at N = 256, K = 512: 1200
    output tiles, several per CTA (the single accumulator handed between
    tiles many times); 64 oracle points per non-empty group, empty groups'
    blocks zero over a NaN sentinel."""
    rng = np.random.default_rng(301)
    sizes = rng.integers(1, 80, size=300)
    sizes[[0, 1, 2, 57, 150, 151, 299]] = 0
    G, N, K = len(sizes), 256, 512
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt = int(off[-1])
    qd = orc.mx_quantize(bits(gen_x((Mt, N), seed=43)), 1, fp8.LAYOUT_COLT, offsets=off, align=128)
    qx = orc.mx_quantize(bits(gen_x((Mt, K), seed=44)), 0, fp8.LAYOUT_COLT, offsets=off, align=128)
    P = qd["q_colT"].shape[1]
    sentinel = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = fp8.mx_grouped_gemm(fp8.GROUPED_K, up(qd["q_colT"]), 1, up(mx_tiled(qd["s_col"])), up(qx["q_colT"]), 0,
                            up(mx_tiled(qx["s_col"])), up(off), Mt, N, K, ld_T=P, out=sentinel)
    assert fp8.fp8_sync_status() == 0
    poff = orc.padded_offsets_align(off, 128)
    out = C.float().cpu().numpy()
    for e in range(G):
        if sizes[e] == 0:
            assert (out[e] == 0).all(), f"empty group {e}"
            continue
        a, b = int(poff[e]), int(poff[e + 1])
        pn, pk = rng.integers(0, N, size=64), rng.integers(0, K, size=64)
        ref, bound = orc.mx_gemm(qd["q_colT"][:, a:b], 1, qd["s_col"][:, a // 32:b // 32],
                                 qx["q_colT"][:, a:b], 0, qx["s_col"][:, a // 32:b // 32], points=(pn, pk))
        check_gemm(out[e][pn, pk], ref, bound, f"kgroup many e{e}")


@pytest.mark.parametrize("K", [256, 160])
def test_mx_grouped_m_bt_small(orc, K):
    """dgrad on the weights' transposed layout: the weight stack [G*K][N]
    MX-quantized in G groups of K rows; expert e's block starts at column
    e * roundup(K, 128) of the transposed layout."""
    sizes = [5, 0, 200, 1, 0, 129, 64]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mt, N = int(off[-1]), 320
    xa = gen_x((Mt, K), seed=51)
    qa = orc.mx_quantize(bits(xa), 1, fp8.LAYOUT_ROW, offsets=off, align=128)
    woff = (np.arange(G + 1) * K).astype(np.int32)
    qw = orc.mx_quantize(bits(gen_x((G * K, N), seed=52)), 0, fp8.LAYOUT_COLT, offsets=woff, align=128)
    kpad = -(-K // 128) * 128
    P = qw["q_colT"].shape[1]
    assert P == G * kpad
    C = fp8.mx_grouped_gemm(fp8.GROUPED_M_BT, up(qa["q_row"]), 1, up(mx_tiled(qa["s_row"])), up(qw["q_colT"]), 0,
                            up(mx_tiled(qw["s_col"])), up(off), Mt, N, K, ld_T=P)
    assert fp8.fp8_sync_status() == 0
    poff = orc.padded_offsets_align(off, 128)
    out = C.float().cpu().numpy()
    for e in range(G):
        if sizes[e] == 0:
            continue
        r0, r1 = off[e], off[e + 1]
        c0 = e * kpad
        ref, bound = orc.mx_gemm(qa["q_row"][r0:r1], 1, qa["s_row"][poff[e]:poff[e] + sizes[e]],
                                 qw["q_colT"][:, c0:c0 + K], 0, qw["s_col"][:, c0 // 32:(c0 + K) // 32])
        check_gemm(out[r0:r1], ref, bound, f"m_bt e{e}")


def test_mx_grouped_bad_offsets_flagged():
    off = torch.tensor([0, 50, 20, 64], dtype=torch.int32, device=DEV)
    A = torch.zeros((64, 128), dtype=torch.uint8, device=DEV)
    B = torch.zeros((3 * 256, 128), dtype=torch.uint8, device=DEV)
    s = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    C = torch.full((64, 256), 3.0, dtype=torch.bfloat16, device=DEV)
    fp8.fp8_mx_grouped_gemm(fp8.GROUPED_M, A, 0, s, B, 0, s, off, 3, 64, 256, 128, C)
    assert fp8.fp8_sync_status() == 1
    assert (C == 3.0).all()


def test_mx_quantize_equal_groups_is_plain():
    """Groups of equal size that are multiples of 128 rows (a stack of expert
    weights) have no padding, so the grouped MX quantize equals the plain
    one on the whole stack: bytes and scale bytes."""
    E, m, cols = 8, 256, 160
    x = gen_x((E * m, cols), seed=31).to(DEV)
    off = np.arange(E + 1, dtype=np.int32) * m
    for fmt in (0, 1):
        qg = fp8.mx_quantize(x, fmt, 3, group_offsets=torch.from_numpy(off).to(DEV), host_offsets=off)
        qp = fp8.mx_quantize(x, fmt, 3)
        assert fp8.fp8_sync_status() == 0
        assert qg.scale_rows == qp.scale_rows == E * m
        assert torch.equal(qg.q_row, qp.q_row) and torch.equal(qg.s_row, qp.s_row)
        assert torch.equal(qg.q_colT[:, :E * m], qp.q_colT[:, :E * m]) and torch.equal(qg.s_col, qp.s_col)
