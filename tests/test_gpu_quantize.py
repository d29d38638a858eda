"""GPU parity of fp8_quantize and fp8_update_amax_history against the oracle.

Bytes, scale_inv values, amaxes and history rows must match bit for bit (NaN
outputs by class).  Sizes span several tiles plus ragged tails; the
full-size cases use the Llama-3-8B / DeepSeek-V3 shapes with full or sampled
checks.
"""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import assert_codes_equal, assert_f32_bits_equal, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    fp8.load_library()


def gen_x(shape, seed, scale=1.0, outliers=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    if outliers and x.numel() > 10:
        idx = torch.randperm(x.numel(), generator=g)[: max(1, x.numel() // 1000)]
        x.view(-1)[idx] *= 50
    return x.to(torch.bfloat16)


def run_gpu(x, fmt, kind, layouts=3, scale=None, amax0=0.0, margin=0, offsets=None):
    xd = x.to(DEV)
    rec = fp8.Recipe(kind=kind, margin=margin)
    scale_in = torch.tensor([scale if scale is not None else 1.0], dtype=torch.float32, device=DEV)
    amax = torch.tensor([amax0], dtype=torch.float32, device=DEV)
    off_d = None if offsets is None else torch.as_tensor(offsets, dtype=torch.int32).to(DEV)
    q = fp8.quantize(xd, fmt, rec, layouts, scale_in=scale_in if kind == fp8.DELAYED else None,
                     amax_out=amax if kind != fp8.ROWWISE else amax, group_offsets=off_d,
                     host_offsets=offsets)
    assert fp8.fp8_sync_status() == 0
    return q, float(amax.cpu()[0])


def compare(orc, x, fmt, kind, layouts=3, scale=None, amax0=0.0, margin=0, offsets=None, what=""):
    q, amax = run_gpu(x, fmt, kind, layouts, scale, amax0, margin, offsets)
    ref = orc.quantize(bits(x), fmt, kind, margin=margin, layouts=layouts,
                       scale_in=np.float32(scale if scale is not None else 1.0), amax_io=np.float32(amax0),
                       offsets=offsets)
    rows = x.shape[0]
    if layouts & 1:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, what + " q_row")
        assert_f32_bits_equal(q.scale_inv_row.cpu().numpy(), ref["scale_inv_row"], what + " sinv_row")
    if layouts & 2:
        ldT = ref["q_colT"].shape[1]
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :ldT], ref["q_colT"], fmt, what + " q_colT")
        assert_f32_bits_equal(q.scale_inv_col.cpu().numpy().ravel(), ref["scale_inv_col"].ravel(),
                              what + " sinv_col")
    assert_f32_bits_equal(np.array([amax], np.float32), np.array([ref["amax"]], np.float32), what + " amax")
    return q, ref


SHAPES = [(1, 8), (37, 136), (128, 128), (129, 256), (300, 520), (256, 512), (1000, 1032)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_quantize_small(orc, shape, fmt, kind):
    x = gen_x(shape, seed=shape[0] * 7 + shape[1] + fmt + 10 * kind, scale=0.3 if fmt == 0 else 1e-3)
    compare(orc, x, fmt, kind, scale=37.5 if fmt == 0 else 2.0 ** 20, amax0=0.25, what=f"{shape} f{fmt} k{kind}")


@pytest.mark.parametrize("layouts", [1, 2])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_quantize_single_layout(orc, layouts, kind):
    x = gen_x((257, 392), seed=5 + layouts + kind)
    compare(orc, x, 0, kind, layouts=layouts, scale=100.0, what=f"layouts {layouts}")


def test_quantize_margin(orc):
    x = gen_x((130, 264), seed=77)
    for m in (1, 3):
        compare(orc, x, 0, 2, margin=m, what=f"margin {m}")
        compare(orc, x, 1, 1, margin=m, what=f"margin {m}")


def test_quantize_special_values(orc):
    g = torch.Generator().manual_seed(3)
    x = synth.randomize_special(gen_x((200, 264), seed=9), g, frac=0.02)
    x[5, :] = 0.0                           # all-zero row
    x[:, 17] = 0.0                          # all-zero column
    x[7, 3] = float("nan")
    x[9, 4] = float("inf")
    x[11, 5] = -float("inf")
    for kind in (0, 1, 2):
        for fmt in (0, 1):
            compare(orc, x, fmt, kind, scale=3.0, what=f"special k{kind} f{fmt}")


def test_quantize_saturation_and_tiny_scale(orc):
    x = gen_x((64, 128), seed=12, scale=1e3)
    compare(orc, x, 0, 0, scale=1e4, what="saturating delayed")          # most values saturate
    compare(orc, x, 1, 0, scale=1e-30, what="underflow delayed")         # everything underflows


def test_quantize_empty(orc):
    x = torch.zeros((0, 64), dtype=torch.bfloat16)
    for kind in (0, 1, 2):
        q, amax = run_gpu(x, 0, kind, layouts=3, scale=4.0, amax0=0.5)
        if kind == 0:
            assert amax == 0.5 and q.scale_inv_row.cpu()[0] == np.float32(0.25)
        else:
            assert amax == 0.0
        if kind == 2:
            assert torch.all(q.scale_inv_col.cpu() == 1.0)


def test_quantize_strided_input(orc):
    base = gen_x((150, 400), seed=21)
    xd = base.to(DEV)[:, :264]               # ld_x = 400 > cols
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    q = fp8.quantize(xd, 0, rec, 3)
    ref = orc.quantize(bits(base[:, :264].contiguous()), 0, 2)
    assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], 0, "strided q_row")
    assert_codes_equal(q.q_colT.cpu().numpy()[:, :150], ref["q_colT"], 0, "strided q_colT")


GROUP_CASES = [
    [5, 0, 33, 1, 0, 40, 128, 200],
    [0, 0, 64],
    [1],
    [31, 32, 33, 0, 95, 96, 97],
]


@pytest.mark.parametrize("sizes", GROUP_CASES)
@pytest.mark.parametrize("kind", [0, 2])
def test_quantize_grouped(orc, sizes, kind):
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = gen_x((int(off[-1]), 136), seed=len(sizes) + kind)
    q, ref = compare(orc, x, 1, kind, scale=512.0, offsets=off, what=f"grouped {sizes}")
    # the padded tail beyond the last group is never written; the oracle's
    # layout ends exactly at the padded total
    assert q.ld_colT >= ref["q_colT"].shape[1]


@pytest.mark.parametrize("layouts", [1, 2])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_quantize_grouped_single_layout(orc, layouts, kind):
    """One layout at a time, every recipe, groups that straddle the cast
    pass's 128-row tiles (sizes 0-200, 72 columns: one full and one partial
    64-column chunk)."""
    sizes = [5, 0, 33, 1, 0, 40, 128, 200, 97]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = gen_x((int(off[-1]), 72), seed=7 + kind + layouts)
    compare(orc, x, 0, kind, layouts=layouts, scale=96.0, offsets=off, what=f"grouped layouts {layouts} kind {kind}")


def test_grouped_bad_offsets_reported():
    x = gen_x((40, 64), seed=1).to(DEV)
    off = torch.tensor([0, 30, 20, 40], dtype=torch.int32, device=DEV)   # decreasing: malformed
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    fp8.quantize(x, 0, rec, 3, group_offsets=off, host_offsets=[0, 30, 30, 40])
    assert fp8.fp8_sync_status() == 1     # FP8_ERR_INVALID_ARG from the device word
    assert fp8.fp8_sync_status() == 0     # cleared


# --- history update ----------------------------------------------------------

def gpu_update(hist, scale, sinv, fmt, algo, margin, cnt):
    h = torch.from_numpy(hist).to(DEV)
    s = torch.from_numpy(scale).to(DEV)
    si = torch.from_numpy(sinv).to(DEV)
    f = torch.from_numpy(np.asarray(fmt, np.uint8)).to(DEV)
    c = torch.from_numpy(cnt).to(DEV)
    fp8.fp8_update_amax_history(h, s, si, f, hist.shape[0], hist.shape[1], algo, margin, c)
    assert fp8.fp8_sync_status() == 0
    return h.cpu().numpy(), s.cpu().numpy(), si.cpu().numpy(), c.cpu().numpy()


@pytest.mark.parametrize("L", [1, 4, 1024, 4096, 32768])
@pytest.mark.parametrize("algo", [0, 1])
def test_update_matches_oracle(orc, L, algo):
    rng = np.random.default_rng(L + algo)
    n = 9
    hist = rng.lognormal(0, 3, size=(n, L)).astype(np.float32)
    hist[1, 0] = 0.0
    hist[2, L // 2] = np.inf
    hist[3, 0] = np.nan
    hist[4, :] = 0.0
    hist[5, 0] = 1e-44                       # scale overflows -> FLT_MAX
    fmt = np.array([0, 1, 0, 1, 0, 3, 1, 2, 3], np.uint8)
    scale = rng.uniform(0.5, 2, n).astype(np.float32)
    sinv = (1 / scale).astype(np.float32)
    cnt = np.zeros(n, np.int32)
    gh, gs, gsi, gc = gpu_update(hist, scale, sinv, fmt, algo, 1, cnt)
    rh, rs, rsi, rc = hist.copy(), scale.copy(), sinv.copy(), cnt.copy()
    orc.update_amax_history(rh, rs, rsi, fmt, algo, 1, rc)
    assert_f32_bits_equal(gh, rh, "hist")
    assert_f32_bits_equal(gs, rs, "scale")
    assert_f32_bits_equal(gsi, rsi, "scale_inv")
    assert np.array_equal(gc, rc)


def test_update_multi_step_sequence(orc):
    """Quantize -> update for 20 steps on the GPU and in the oracle (delayed, max)."""
    L, n = 16, 3
    rng = np.random.default_rng(4)
    hist_d = torch.zeros((n, L), dtype=torch.float32, device=DEV)
    scale_d = torch.ones(n, dtype=torch.float32, device=DEV)
    sinv_d = torch.ones(n, dtype=torch.float32, device=DEV)
    fmt_np = np.array([0, 0, 1], np.uint8)
    fmt_d = torch.from_numpy(fmt_np).to(DEV)
    hist_o = np.zeros((n, L), np.float32)
    scale_o = np.ones(n, np.float32)
    sinv_o = np.ones(n, np.float32)
    rec = fp8.Recipe(kind=fp8.DELAYED)
    for step in range(20):
        for i in range(n):
            x = gen_x((96, 136), seed=100 * step + i, scale=float(rng.lognormal(0, 2)))
            xd = x.to(DEV)
            q = fp8.quantize(xd, int(fmt_np[i]), rec, 3, scale_in=scale_d[i:i + 1], amax_out=hist_d[i, 0:1])
            ref = orc.quantize(bits(x), int(fmt_np[i]), orc.DELAYED, scale_in=scale_o[i], amax_io=hist_o[i, 0])
            hist_o[i, 0] = ref["amax"]
            assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], int(fmt_np[i]), f"step {step} t{i}")
        fp8.fp8_update_amax_history(hist_d, scale_d, sinv_d, fmt_d, n, L, fp8.MAX, 0)
        orc.update_amax_history(hist_o, scale_o, sinv_o, fmt_np, orc.MAX, 0)
        assert_f32_bits_equal(hist_d.cpu().numpy(), hist_o, f"hist step {step}")
        assert_f32_bits_equal(scale_d.cpu().numpy(), scale_o, f"scale step {step}")
        assert_f32_bits_equal(sinv_d.cpu().numpy(), sinv_o, f"sinv step {step}")


def test_bounded_wait_reports_timeout():
    assert fp8.fp8_sync_status() == 0
    assert fp8.fp8_selftest_bounded_wait(2_000_000) == 0   # 2 ms
    assert fp8.fp8_sync_status() == 5                        # FP8_ERR_TIMEOUT
    assert fp8.fp8_sync_status() == 0                        # cleared; the context is still usable
    x = gen_x((64, 64), seed=0).to(DEV)
    fp8.quantize(x, 0, fp8.Recipe(kind=fp8.ROWWISE), 3)
    assert fp8.fp8_sync_status() == 0


def test_deterministic_repeats():
    x = gen_x((700, 1032), seed=8).to(DEV)
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    a = fp8.quantize(x, 0, rec, 3)
    b = fp8.quantize(x, 0, rec, 3)
    # columns past `rows` of the transposed layout are padding the kernel never writes
    assert torch.equal(a.q_row, b.q_row) and torch.equal(a.q_colT[:, :700], b.q_colT[:, :700])
    assert torch.equal(a.scale_inv_col, b.scale_inv_col)


def test_guard_canary():
    """Outputs inside larger buffers: bytes around them stay untouched."""
    x = gen_x((130, 136), seed=31).to(DEV)
    rows, cols, ld = 130, 136, 144
    qrow_buf = torch.full((rows * cols + 64,), 0xA5, dtype=torch.uint8, device=DEV)
    qcol_buf = torch.full((cols * ld + 64,), 0x5A, dtype=torch.uint8, device=DEV)
    sr = torch.full((rows + 8,), -7.0, device=DEV)
    sc = torch.full((cols + 8,), -7.0, device=DEV)
    amax = torch.zeros(1, device=DEV)
    fp8.fp8_quantize(x, rows, cols, cols, 0, fp8.Recipe(kind=fp8.ROWWISE), 3, None, amax, qrow_buf[32:],
                     sr[4:], qcol_buf[32:], ld, sc[4:])
    assert fp8.fp8_sync_status() == 0
    assert torch.all(qrow_buf[:32] == 0xA5) and torch.all(qrow_buf[32 + rows * cols:] == 0xA5)
    assert torch.all(qcol_buf[:32] == 0x5A) and torch.all(qcol_buf[32 + cols * ld:] == 0x5A)
    # ungrouped: the columns rows..ld-1 of each transposed row are left alone
    qc = qcol_buf[32:32 + cols * ld].view(cols, ld)
    assert torch.all(qc[:, rows:] == 0x5A)
    assert torch.all(sr[:4] == -7) and torch.all(sr[4 + rows:] == -7)
    assert torch.all(sc[:4] == -7) and torch.all(sc[4 + cols:] == -7)


# --- full-size shapes -----------------------------------------------------------

def test_full_llama_x_delayed_bitexact(orc):
    """X [8192, 4096] and W_gate [14336, 4096], delayed e4m3: every byte."""
    base = synth.llama_mlp_base()
    for key, scale in (("x", 60.0), ("w_gate", 4000.0)):
        x = base[key]
        compare(orc, x, 0, 0, scale=scale, amax0=0.0, what=key)


def test_full_llama_dy_rowwise_bitexact(orc):
    """dY [8192, 4096] rowwise + colwise e5m2 (config of the rowwise recipe)."""
    x = synth.llama_mlp_base()["dy_down"]
    compare(orc, x, 1, 2, what="dy_down rowwise")


def test_full_moe_tokens_grouped_sampled(orc):
    """Permuted tokens [32768, 7168], rowwise + per-group colwise, sampled."""
    sizes = synth.moe_group_sizes().numpy()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = synth.moe_tokens()["xp"]
    q, _ = run_gpu(x, 0, 2, offsets=off)
    poff = orc.padded_offsets(off)
    g = torch.Generator().manual_seed(0)
    xb = bits(x)
    # sampled rows: the row scale depends on the row only
    for r in torch.randint(0, x.shape[0], (48,), generator=g).tolist():
        ref = orc.quantize(xb[r:r + 1], 0, orc.ROWWISE, layouts=1)
        assert_codes_equal(q.q_row[r:r + 1].cpu().numpy(), ref["q_row"], 0, f"row {r}")
        assert_f32_bits_equal(q.scale_inv_row[r:r + 1].cpu().numpy(), ref["scale_inv_row"], f"srow {r}")
    # every group (empty ones included) for a sample of column blocks
    sc = q.scale_inv_col.view(len(sizes), -1)
    for c0 in (0, 1024, 7160):
        for e in range(len(sizes)):
            r0, r1 = off[e], off[e + 1]
            seg = q.q_colT[c0:c0 + 8, poff[e]:poff[e + 1]].cpu().numpy()
            if r1 == r0:
                assert np.all(sc[e, c0:c0 + 8].cpu().numpy() == 1.0)
                continue
            ref = orc.quantize(xb[r0:r1, c0:c0 + 8], 0, orc.ROWWISE, layouts=2)
            assert_codes_equal(seg[:, :r1 - r0], ref["q_colT"], 0, f"group {e} col {c0}")
            assert not seg[:, r1 - r0:].any()
            assert_f32_bits_equal(sc[e, c0:c0 + 8].cpu().numpy(), ref["scale_inv_col"], f"scol {e} {c0}")


def test_quantize_grouped_large(orc):
    """A large grouped tensor (20000 x 4096, 40 groups incl. empty ones), every byte."""
    g = torch.Generator().manual_seed(41)
    sizes = torch.randint(0, 900, (40,), generator=g).numpy()
    sizes[[3, 17]] = 0
    sizes[-1] = 20000 - sizes[:-1].sum()
    assert sizes[-1] > 0
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = gen_x((int(off[-1]), 4096), seed=42)
    compare(orc, x, 0, 2, offsets=off, what="grouped multi-chunk")


@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
@pytest.mark.parametrize("scale", [1.0, 3.5, 2.0 ** -20, 448.0 / 3.0, 1e30])
def test_cast_every_bf16_pattern(orc, fmt, scale):
    """Every bf16 bit pattern (NaN, Inf, subnormals, both zeros included),
    cast with a stored scale, against the oracle's element-wise encoder."""
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(512, 128)
    q, _ = run_gpu(pats, fmt, 0, scale=scale)
    exp = orc.cast_points(bits(pats), np.float32(scale), fmt).reshape(512, 128)
    assert_codes_equal(q.q_row.cpu().numpy(), exp, fmt, f"patterns f{fmt} s{scale}")
    assert_codes_equal(q.q_colT.cpu().numpy()[:, :512], exp.T, fmt, f"patterns colT f{fmt} s{scale}")


@pytest.mark.parametrize("fmt", [2, 3])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("shape", [(37, 136), (300, 520)])
def test_quantize_fnuz(orc, fmt, kind, shape):
    """e4m3fnuz (max 240) and e5m2fnuz (max 57344): no negative zero, single
    NaN, for every recipe."""
    x = gen_x(shape, seed=shape[0] + kind, scale=0.5)
    compare(orc, x, fmt, kind, scale=100.0, amax0=0.1, what=f"fnuz{fmt} {shape} k{kind}")


@pytest.mark.parametrize("fmt", [2, 3])
def test_quantize_fnuz_grouped_and_special(orc, fmt):
    g = torch.Generator().manual_seed(8)
    x = synth.randomize_special(gen_x((120, 136), seed=10), g, frac=0.03)
    x[3, 5] = float("nan")
    for kind in (0, 1, 2):
        compare(orc, x, fmt, kind, scale=7.0, what=f"fnuz{fmt} special k{kind}")
    sizes = [5, 0, 33, 1, 0, 40]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    compare(orc, gen_x((int(off[-1]), 136), seed=12), fmt, 2, offsets=off, what=f"fnuz{fmt} grouped")


def test_e5m2fnuz_top_binade(orc):
    """Every bf16 value of e5m2fnuz's top binades (|v| in [2^13, 2^17)), the
    range where the GPU encoder switches from e5m2(2v) to e5m2(v/2), plus the
    saturation band above 57344."""
    mags = torch.arange(0x4600, 0x4800, dtype=torch.int32)          # bf16 patterns 2^13 .. 2^17
    pats = torch.cat([mags, mags | 0x8000]).to(torch.int16).view(torch.bfloat16).reshape(8, 128)
    for scale in (1.0, 0.5, 2.0):
        q, _ = run_gpu(pats, 3, 0, scale=scale)
        exp = orc.cast_points(bits(pats), np.float32(scale), 3).reshape(8, 128)
        assert_codes_equal(q.q_row.cpu().numpy(), exp, 3, f"top binade s{scale}")


@pytest.mark.parametrize("layouts", [1, 2, 3])
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_quantize_equal_groups(orc, layouts, fmt):
    """Equal groups without offsets (a stack of 6 expert weights of 128 rows,
    136 columns): the same bytes and scales as the same call with the
    offsets e * 128, and as the oracle's grouped quantize."""
    E, m, cols = 6, 128, 136
    x = gen_x((E * m, cols), seed=60 + fmt + 3 * layouts)
    off = np.arange(E + 1, dtype=np.int32) * m
    rec = fp8.Recipe(kind=fp8.ROWWISE, margin=1)
    xd = x.to(DEV)
    qe = fp8.quantize(xd, fmt, rec, layouts, equal_groups=E)
    qo = fp8.quantize(xd, fmt, rec, layouts, group_offsets=torch.from_numpy(off).to(DEV), host_offsets=off)
    assert fp8.fp8_sync_status() == 0
    ref = orc.quantize(bits(x), fmt, orc.ROWWISE, margin=1, layouts=layouts, offsets=off)
    rows = E * m
    if layouts & 1:
        assert torch.equal(qe.q_row, qo.q_row)
        assert torch.equal(qe.scale_inv_row.view(torch.int32), qo.scale_inv_row.view(torch.int32))
        assert_codes_equal(qe.q_row.cpu().numpy(), ref["q_row"], fmt, "equal groups q_row")
        assert_f32_bits_equal(qe.scale_inv_row.cpu().numpy(), ref["scale_inv_row"], "equal groups sinv_row")
    if layouts & 2:
        assert torch.equal(qe.q_colT[:, :rows], qo.q_colT[:, :rows])
        assert torch.equal(qe.scale_inv_col.view(torch.int32), qo.scale_inv_col.view(torch.int32))
        assert_codes_equal(qe.q_colT.cpu().numpy()[:, :rows], ref["q_colT"], fmt, "equal groups q_colT")
        assert_f32_bits_equal(qe.scale_inv_col.cpu().numpy().reshape(E, cols), ref["scale_inv_col"],
                              "equal groups sinv_col")


def test_quantize_equal_groups_moe_weight():
    """A reduced DeepSeek-V3 gate weight stack (64 experts x 2048 rows x
    7168): equal-groups mode byte-equal to the offsets mode."""
    E, m, cols = 64, 2048, 7168
    g = torch.Generator(device=DEV).manual_seed(7)
    x = (torch.randn((E * m, cols), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    off = np.arange(E + 1, dtype=np.int32) * m
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    qe = fp8.quantize(x, 0, rec, equal_groups=E)
    qo = fp8.quantize(x, 0, rec, group_offsets=torch.from_numpy(off).to(DEV), host_offsets=off)
    assert fp8.fp8_sync_status() == 0
    assert torch.equal(qe.q_row, qo.q_row)
    assert torch.equal(qe.q_colT[:, :E * m], qo.q_colT[:, :E * m])
    assert torch.equal(qe.scale_inv_row.view(torch.int32), qo.scale_inv_row.view(torch.int32))
    assert torch.equal(qe.scale_inv_col.view(torch.int32), qo.scale_inv_col.view(torch.int32))


@pytest.mark.parametrize("groups", [0, 40, 2560])
def test_quantize_rowwise_tall(orc, groups):
    """A tall tensor (163840 x 160, the last column chunk ragged): every
    block's run of tiles in the amax pass spans several row blocks, and with
    40 equal groups of 4096 rows many runs cross a group boundary (2560 groups
    of 64 rows: every row block starts a group); bytes and scales bit-exact
    against the oracle."""
    rows, cols, fmt = 163840, 160, 1
    x = gen_x((rows, cols), seed=71 + groups)
    off = np.arange(groups + 1, dtype=np.int32) * (rows // groups) if groups else None
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    q = fp8.quantize(x.to(DEV), fmt, rec, 3, equal_groups=groups)
    assert fp8.fp8_sync_status() == 0
    ref = orc.quantize(bits(x), fmt, orc.ROWWISE, layouts=3, offsets=off)
    what = f"tall, {groups} groups"
    assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, f"{what} q_row")
    assert_f32_bits_equal(q.scale_inv_row.cpu().numpy(), ref["scale_inv_row"], f"{what} sinv_row")
    assert_codes_equal(q.q_colT.cpu().numpy()[:, :rows], ref["q_colT"], fmt, f"{what} q_colT")
    sc = q.scale_inv_col.cpu().numpy()
    assert_f32_bits_equal(sc.reshape(groups, cols) if groups else sc, ref["scale_inv_col"], f"{what} sinv_col")
