"""GPU parity of fp8_scaled_gemm and fp8_grouped_gemm against the oracle.

Tolerance (elementwise): |out - ref| <= 2e-3 * sum_k |a_k b_k sa sb| + 1e-5,
with ref the oracle's fp64 dequantised product.  Small shapes are compared
in full (several tiles plus ragged M / N / K tails); the Llama-3-8B and
DeepSeek-V3 shapes on 64 full rows, 64 full columns and 4096 random points.
"""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import check_gemm, finite_codes, realistic_codes, sample_points

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    fp8.load_library()


def run_gemm(A, fa, B, fb, sa, sb, K=None):
    C = fp8.scaled_gemm(A.to(DEV), fa, B.to(DEV), fb, sa.to(DEV), sb.to(DEV), K=K)
    assert fp8.fp8_sync_status() == 0
    return C


def scales(g, n, per_row):
    if per_row:
        return (torch.rand(n, generator=g) * 2 + 0.01).to(torch.float32)
    return torch.tensor([float(torch.rand(1, generator=g)) + 0.5], dtype=torch.float32)


SMALL = [(128, 256, 128), (1, 8, 16), (100, 40, 48), (130, 300, 144), (256, 512, 512), (300, 520, 1040),
         (129, 257, 4096)]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
@pytest.mark.parametrize("per_row", [False, True])
def test_gemm_small_full(orc, shape, fa, fb, per_row):
    M, N, K = shape
    g = torch.Generator().manual_seed(M * 3 + N + K + fa * 2 + fb + per_row)
    A = finite_codes(g, (M, K), fa)
    B = finite_codes(g, (N, K), fb)
    sa, sb = scales(g, M, per_row), scales(g, N, per_row)
    C = run_gemm(A, fa, B, fb, sa, sb)
    ref, bound = orc.gemm(A.numpy(), fa, B.numpy(), fb, sa.numpy(), sb.numpy())
    check_gemm(C.float().cpu().numpy(), ref, bound, f"{shape}")


def test_gemm_realistic_values(orc):
    g = torch.Generator().manual_seed(11)
    M, N, K = 384, 768, 2048
    A = realistic_codes(g, (M, K), 0)
    B = realistic_codes(g, (N, K), 1)
    sa, sb = scales(g, M, True), scales(g, N, True)
    C = run_gemm(A, 0, B, 1, sa, sb)
    ref, bound = orc.gemm(A.numpy(), 0, B.numpy(), 1, sa.numpy(), sb.numpy())
    check_gemm(C.float().cpu().numpy(), ref, bound, "realistic", strict=True)


def test_gemm_padded_leading_dims(orc):
    """A and B inside wider buffers (lda, ldb > K); C with ldc > N."""
    g = torch.Generator().manual_seed(5)
    M, N, K = 200, 264, 160
    Ab = finite_codes(g, (M, 256), 0)
    Bb = finite_codes(g, (N, 192), 0)
    sa, sb = scales(g, M, True), scales(g, 1, False)
    Cb = torch.full((M, 272), 7.0, dtype=torch.bfloat16, device=DEV)
    fp8.fp8_scaled_gemm(Ab.to(DEV), 0, 256, Bb.to(DEV), 0, 192, M, N, K, sa.to(DEV), 1, sb.to(DEV), 0, Cb, 272)
    assert fp8.fp8_sync_status() == 0
    ref, bound = orc.gemm(Ab[:, :K].numpy(), 0, Bb[:, :K].numpy(), 0, sa.numpy(), sb.numpy())
    out = Cb.float().cpu().numpy()
    check_gemm(out[:, :N], ref, bound, "padded")
    assert np.all(out[:, N:] == 7.0)   # columns past N untouched


def test_gemm_special_operands(orc):
    M, N, K = 256, 256, 256
    A = torch.zeros((M, K), dtype=torch.uint8)
    for i in range(M):
        A[i, i % K] = 0x38                      # one-hot rows of 1.0
    g = torch.Generator().manual_seed(2)
    B = finite_codes(g, (N, K), 0)
    sa = torch.tensor([1.0]); sb = torch.tensor([1.0])
    C = run_gemm(A, 0, B, 0, sa, sb)
    ref, bound = orc.gemm(A.numpy(), 0, B.numpy(), 0, sa.numpy(), sb.numpy())
    check_gemm(C.float().cpu().numpy(), ref, bound, "one-hot")
    Z = run_gemm(torch.zeros((M, K), dtype=torch.uint8), 0, B, 0, sa, sb)
    assert torch.all(Z == 0)


def test_gemm_deterministic(orc):
    g = torch.Generator().manual_seed(3)
    A = finite_codes(g, (512, 1024), 0).to(DEV)
    B = finite_codes(g, (768, 1024), 0).to(DEV)
    sa = torch.ones(1, device=DEV); sb = torch.ones(1, device=DEV)
    c1 = fp8.scaled_gemm(A, 0, B, 0, sa, sb)
    c2 = fp8.scaled_gemm(A, 0, B, 0, sa, sb)
    assert torch.equal(c1, c2)


def _sampled(orc, M, N, K, fa, fb, seed, per_row=True):
    gd = torch.Generator(device=DEV).manual_seed(seed)
    xa = torch.randn((M, K), generator=gd, device=DEV)
    xb = torch.randn((N, K), generator=gd, device=DEV)
    dta = torch.float8_e4m3fn if fa == 0 else torch.float8_e5m2
    dtb = torch.float8_e4m3fn if fb == 0 else torch.float8_e5m2
    # torch's cast is not saturating: clamp to the format range first
    A = (xa * 100).clamp(-448, 448).to(dta).view(torch.uint8)
    B = (xb * 100).clamp(-448, 448).to(dtb).view(torch.uint8)
    del xa, xb
    g = torch.Generator().manual_seed(seed)
    sa, sb = scales(g, M, per_row), scales(g, N, per_row)
    C = fp8.scaled_gemm(A, fa, B, fb, sa.to(DEV), sb.to(DEV))
    assert fp8.fp8_sync_status() == 0
    pm, pn = sample_points(g, M, N)
    out = C[torch.from_numpy(pm).to(DEV), torch.from_numpy(pn).to(DEV)].float().cpu().numpy()
    ref, bound = orc.gemm(A.cpu().numpy(), fa, B.cpu().numpy(), fb, sa.numpy(), sb.numpy(), points=(pm, pn))
    return check_gemm(out, ref, bound, f"{M}x{N}x{K}", strict=True)


def test_gemm_llama_gate_fprop_sampled(orc):
    _sampled(orc, 8192, 14336, 4096, 0, 0, seed=1)


def test_gemm_llama_down_fprop_sampled(orc):
    _sampled(orc, 8192, 4096, 14336, 0, 0, seed=2, per_row=False)


def test_gemm_llama_wgrad_sampled(orc):
    _sampled(orc, 14336, 4096, 8192, 1, 0, seed=3)


# --- grouped ----------------------------------------------------------------------

def offsets_of(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


@pytest.mark.parametrize("sizes", [[5, 0, 33, 1, 0, 140, 128, 300], [0, 0, 256], [1], [129] * 5])
@pytest.mark.parametrize("per_row", [True, False])
def test_grouped_m_small(orc, sizes, per_row):
    off = offsets_of(sizes)
    G, Mt, N, K = len(sizes), int(off[-1]), 264, 272
    g = torch.Generator().manual_seed(sum(sizes) + per_row)
    A = finite_codes(g, (Mt, K), 0)
    B = finite_codes(g, (G, N, K), 0)
    sa = scales(g, Mt, per_row)
    sb = scales(g, G * N, per_row)
    C = torch.full((max(Mt, 1), N), 3.0, dtype=torch.bfloat16, device=DEV)
    fp8.grouped_gemm(fp8.GROUPED_M, A.to(DEV), 0, B.to(DEV), 0, torch.from_numpy(off).to(DEV), Mt, N, K,
                     sa.to(DEV), sb.to(DEV), out=C[:Mt] if Mt else C)
    assert fp8.fp8_sync_status() == 0
    if Mt == 0:
        return
    pm, pn = np.meshgrid(np.arange(Mt), np.arange(N), indexing="ij")
    ref, bound = orc.grouped_gemm(0, A.numpy(), 0, B.numpy(), 0, off, N, K, sa.numpy(), sb.numpy(), None,
                                  pm.ravel(), pn.ravel())
    check_gemm(C[:Mt].float().cpu().numpy().ravel(), ref, bound, f"grouped M {sizes}")


@pytest.mark.parametrize("sizes", [[5, 0, 33, 1, 0, 140, 128, 300], [0, 0, 256], [1], [200, 0]])
@pytest.mark.parametrize("NK", [(136, 264), (160, 296), (96, 520)])
def test_grouped_k_small(orc, sizes, NK):
    """(136, 264) takes the direct-store epilogue; N % 32 == 0 and K % 8 == 0
    take the TMA-store epilogue (partial 128-row tiles, K ending inside a box)."""
    off = offsets_of(sizes)
    poff = orc.padded_offsets(off)
    ldT = max(16, int(poff[-1]))
    G, (N, K) = len(sizes), NK
    g = torch.Generator().manual_seed(len(sizes) * 13)
    AT = torch.zeros((N, ldT), dtype=torch.uint8)
    BT = torch.zeros((K, ldT), dtype=torch.uint8)
    for e, m in enumerate(sizes):
        AT[:, poff[e]:poff[e] + m] = finite_codes(g, (N, m), 1)
        BT[:, poff[e]:poff[e] + m] = finite_codes(g, (K, m), 0)
    sa = scales(g, G * N, True)
    sb = scales(g, G * K, True)
    # a NaN sentinel in every element: the empty groups' zeros are written, not left over
    sentinel = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = fp8.grouped_gemm(fp8.GROUPED_K, AT.to(DEV), 1, BT.to(DEV), 0, torch.from_numpy(off).to(DEV),
                         int(off[-1]), N, K, sa.to(DEV), sb.to(DEV), ld_T=ldT, out=sentinel)
    assert fp8.fp8_sync_status() == 0
    pg, pn, pk = np.meshgrid(np.arange(G), np.arange(N), np.arange(K), indexing="ij")
    ref, bound = orc.grouped_gemm(1, AT.numpy(), 1, BT.numpy(), 0, off, N, K, sa.numpy(), sb.numpy(),
                                  pg.ravel(), pn.ravel(), pk.ravel())
    out = C.float().cpu().numpy().ravel()
    check_gemm(out, ref, bound, f"grouped K {sizes}")
    for e, m in enumerate(sizes):
        if m == 0:
            assert torch.all(C[e] == 0)


def test_grouped_k_many_tiles_per_cta(orc):
    """300 small groups with runs of empty ones at N = 256, K = 512: 1200
    output tiles, so every CTA takes several in turn and both epilogue
    groups, both accumulators and their phases are exercised; sampled
    against the oracle, and every empty group's block is zero (over a NaN
    sentinel)."""
    rng = np.random.default_rng(300)
    g = torch.Generator().manual_seed(300)
    sizes = rng.integers(1, 80, size=300)
    sizes[[0, 1, 2, 57, 150, 151, 299]] = 0
    off = offsets_of(sizes)
    poff = orc.padded_offsets(off)
    ldT = max(16, int(poff[-1]))
    G, N, K = len(sizes), 256, 512
    AT = torch.zeros((N, ldT), dtype=torch.uint8)
    BT = torch.zeros((K, ldT), dtype=torch.uint8)
    for e, m in enumerate(sizes):
        if m:
            AT[:, poff[e]:poff[e] + m] = finite_codes(g, (N, int(m)), 1)
            BT[:, poff[e]:poff[e] + m] = finite_codes(g, (K, int(m)), 0)
    sa = scales(g, G * N, True)
    sb = scales(g, G * K, True)
    sentinel = torch.full((G, N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = fp8.grouped_gemm(fp8.GROUPED_K, AT.to(DEV), 1, BT.to(DEV), 0, torch.from_numpy(off).to(DEV),
                         int(off[-1]), N, K, sa.to(DEV), sb.to(DEV), ld_T=ldT, out=sentinel)
    assert fp8.fp8_sync_status() == 0
    pg = rng.integers(0, G, size=20000)
    pn = rng.integers(0, N, size=20000)
    pk = rng.integers(0, K, size=20000)
    ref, bound = orc.grouped_gemm(1, AT.numpy(), 1, BT.numpy(), 0, off, N, K, sa.numpy(), sb.numpy(), pg, pn, pk)
    out = C.float().cpu().numpy()
    check_gemm(out[pg, pn, pk], ref, bound, "grouped K, 300 groups")
    for e in np.flatnonzero(sizes == 0):
        assert (out[e] == 0).all(), f"empty group {e}"


def test_grouped_m_moe_shape_sampled(orc):
    """DeepSeek-V3 gate projection: 32768 routed rows, 256 experts, 7168 -> 2048."""
    sizes = synth.moe_group_sizes().numpy()
    off = offsets_of(sizes)
    G, Mt, N, K = len(sizes), int(off[-1]), 2048, 7168
    gd = torch.Generator(device=DEV).manual_seed(9)
    A = (torch.randn((Mt, K), generator=gd, device=DEV) * 100).clamp(-448, 448).to(torch.float8_e4m3fn)
    A = A.view(torch.uint8)
    B = (torch.randn((G, N, K), generator=gd, device=DEV) * 100).clamp(-448, 448).to(torch.float8_e4m3fn)
    B = B.view(torch.uint8)
    g = torch.Generator().manual_seed(9)
    sa = scales(g, Mt, True)
    sb = scales(g, G * N, True)
    C = fp8.grouped_gemm(fp8.GROUPED_M, A, 0, B, 0, torch.from_numpy(off).to(DEV), Mt, N, K, sa.to(DEV),
                         sb.to(DEV))
    assert fp8.fp8_sync_status() == 0
    # sampled experts: largest, smallest non-empty, 8 random
    nz = np.nonzero(sizes)[0]
    experts = {int(np.argmax(sizes)), int(nz[np.argmin(sizes[nz])])}
    experts |= set(torch.randint(0, G, (8,), generator=g).tolist())
    Acpu = A.cpu().numpy()
    for e in sorted(experts):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        rows = np.arange(r0, r1)[torch.randperm(r1 - r0, generator=g)[:16].numpy()]
        pm = np.repeat(rows, N).astype(np.int64)
        pn = np.tile(np.arange(N), len(rows)).astype(np.int64)
        Be = B[e:e + 1].cpu().numpy()
        sub_off = np.array([0, r1 - r0], np.int32)
        ref, bound = orc.grouped_gemm(0, Acpu[r0:r1], 0, Be, 0, sub_off, N, K, sa.numpy()[r0:r1],
                                      sb.numpy()[e * N:(e + 1) * N], None, pm - r0, pn)
        out = C[torch.from_numpy(pm).to(DEV), torch.from_numpy(pn).to(DEV)].float().cpu().numpy()
        check_gemm(out, ref, bound, f"expert {e}")


@pytest.mark.parametrize("sizes,K", [([5, 0, 33, 1, 0, 140, 128, 300], 272), ([64, 0, 200], 80), ([1], 48)])
def test_grouped_m_bt_small(orc, sizes, K):
    """M-grouped with B in the grouped colwise layout of a weight tensor (dgrad)."""
    off = offsets_of(sizes)
    G, Mt, N = len(sizes), int(off[-1]), 264
    kpad = (K + 31) // 32 * 32
    ldT = (G * kpad + 15) // 16 * 16 + 16          # a little wider than needed
    g = torch.Generator().manual_seed(sum(sizes) + K)
    A = finite_codes(g, (Mt, K), 1)
    Bexp = finite_codes(g, (G, N, K), 0)            # expert e: [N][K]
    BT = torch.full((N, ldT), 0x7F, dtype=torch.uint8)   # NaN bytes where no expert data lives
    for e in range(G):
        BT[:, e * kpad:e * kpad + K] = Bexp[e]
        BT[:, e * kpad + K:(e + 1) * kpad] = 0          # zero padding, as fp8_quantize writes it
    sa = scales(g, Mt, True)
    sb = scales(g, G * N, True)
    C = fp8.grouped_gemm(fp8.GROUPED_M_BT, A.to(DEV), 1, BT.to(DEV), 0, torch.from_numpy(off).to(DEV), Mt, N, K,
                         sa.to(DEV), sb.to(DEV), ld_T=ldT)
    assert fp8.fp8_sync_status() == 0
    pm, pn = np.meshgrid(np.arange(Mt), np.arange(N), indexing="ij")
    ref, bound = orc.grouped_gemm(0, A.numpy(), 1, Bexp.numpy(), 0, off, N, K, sa.numpy(), sb.numpy(), None,
                                  pm.ravel(), pn.ravel())
    check_gemm(C.float().cpu().numpy().ravel(), ref, bound, f"grouped M^T {sizes}")
