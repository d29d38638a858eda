"""Whole-workload GPU parity: the five workloads run through the library as a
training step would, checked against the oracle.

  1 tiny FP8 linear, rowwise recipe: every byte, scale and GEMM output.
  2 Llama-3-8B MLP block, delayed scaling (hybrid, most_recent, L = 1024),
    50 steps of drifting scale at full size: history, scale and scale_inv
    bit-exact at every step, amax of every tensor every step, bytes of
    sampled rows / columns every step and every byte of X at steps 0, 30,
    49; the 9 GEMMs within tolerance at steps 0, 1, 30, 49 (sampled).
  3 Llama-3-8B attention projections, rowwise recipe with Student-t
    activations: full bytes / scales of X, sampled for the rest; the six
    GEMMs sampled.
  4 DeepSeek-V3 MoE layer: rowwise + per-group colwise quantize of the
    routed tokens and the expert weights, the nine grouped GEMMs, checked on
    the largest, the smallest non-empty, all empty and 8 random experts.
  5 Flux-12B linears, delayed scaling (all E4M3, amax algo max), 50 drifting
    steps as in 2.
"""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth
from parity import assert_codes_equal, assert_f32_bits_equal, bits, check_gemm

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    fp8.load_library()


def sync_ok():
    assert fp8.fp8_sync_status() == 0


def sampled_gemm_check(orc, A, fa, B, fb, sa, sb, C, seed, what, n_rows=8, n_cols=8, n_rand=2048, strict=False):
    """Check C = A.B^T * sa * sb on sampled full rows, full columns and random
    points (strict: the stated bound alone, for random-sign data at large K)."""
    M, K = A.shape
    N = B.shape[0]
    g = torch.Generator().manual_seed(seed)
    rows = torch.randperm(M, generator=g)[:n_rows].numpy()
    cols = torch.randperm(N, generator=g)[:n_cols].numpy()
    pm = np.concatenate([np.repeat(rows, N), np.tile(np.arange(M), len(cols)),
                         torch.randint(0, M, (n_rand,), generator=g).numpy()]).astype(np.int64)
    pn = np.concatenate([np.tile(np.arange(N), len(rows)), np.repeat(cols, M),
                         torch.randint(0, N, (n_rand,), generator=g).numpy()]).astype(np.int64)
    out = C[torch.from_numpy(pm).to(DEV), torch.from_numpy(pn).to(DEV)].float().cpu().numpy()
    ref, bound = orc.gemm(A.cpu().numpy(), fa, B.cpu().numpy(), fb, sa.cpu().numpy(), sb.cpu().numpy(),
                          points=(pm, pn))
    check_gemm(out, ref, bound, what, strict=strict)


# --------------------------------------------------------------------------------------------
# 1. tiny
# --------------------------------------------------------------------------------------------

def test_config1_tiny_full(orc):
    t = synth.tiny()
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    fmts = {"x": 0, "w": 0, "dy": 1}
    q, r = {}, {}
    for k, f in fmts.items():
        q[k] = fp8.quantize(t[k].to(DEV), f, rec)
        r[k] = orc.quantize(bits(t[k]), f, orc.ROWWISE)
        rows = t[k].shape[0]
        assert_codes_equal(q[k].q_row.cpu().numpy(), r[k]["q_row"], f, k)
        assert_codes_equal(q[k].q_colT.cpu().numpy()[:, :rows], r[k]["q_colT"], f, k)
        assert_f32_bits_equal(q[k].scale_inv_row.cpu().numpy(), r[k]["scale_inv_row"], k)
        assert_f32_bits_equal(q[k].scale_inv_col.cpu().numpy(), r[k]["scale_inv_col"], k)
    sync_ok()
    gemms = {  # name: (A, fa, A layout, B, fb, B layout)
        "fprop": ("x", "row", "w", "row"),
        "dgrad": ("dy", "row", "w", "colT"),
        "wgrad": ("dy", "colT", "x", "colT"),
    }
    for name, (a, al, b, bl) in gemms.items():
        qa = q[a].q_row if al == "row" else q[a].q_colT
        qb = q[b].q_row if bl == "row" else q[b].q_colT
        sa = q[a].scale_inv_row if al == "row" else q[a].scale_inv_col
        sb = q[b].scale_inv_row if bl == "row" else q[b].scale_inv_col
        K = qa.shape[1] if al == "row" else t[a].shape[0]
        C = fp8.scaled_gemm(qa, fmts[a], qb, fmts[b], sa, sb, K=K)
        sync_ok()
        ra = r[a]["q_row"] if al == "row" else r[a]["q_colT"]
        rb = r[b]["q_row"] if bl == "row" else r[b]["q_colT"]
        rsa = r[a]["scale_inv_row"] if al == "row" else r[a]["scale_inv_col"]
        rsb = r[b]["scale_inv_row"] if bl == "row" else r[b]["scale_inv_col"]
        ref, bound = orc.gemm(ra, fmts[a], rb, fmts[b], rsa, rsb)
        check_gemm(C.float().cpu().numpy(), ref, bound, name)


# --------------------------------------------------------------------------------------------
# 2 and 5. delayed scaling over 50 drifting steps
# --------------------------------------------------------------------------------------------

class DelayedLayer:
    """Device buffers of a block of Linears under delayed scaling."""

    def __init__(self, base, fmts, L, algo):
        self.names = list(base)
        self.base = {k: v.to(DEV) for k, v in base.items()}
        self.fmt = fmts
        n = len(self.names)
        self.L, self.algo = L, algo
        self.hist = torch.zeros((n, L), device=DEV)
        self.scale = torch.ones(n, device=DEV)
        self.sinv = torch.ones(n, device=DEV)
        self.fmt_dev = torch.tensor([fmts[k] for k in self.names], dtype=torch.uint8, device=DEV)
        self.rec = fp8.Recipe(kind=fp8.DELAYED, history_len=L, algo=algo)
        self.q = {}
        self.x = {}

    def step_quantize(self, t):
        for i, k in enumerate(self.names):
            self.x[k] = synth.drifted(self.base[k], k, t)
            self.q[k] = fp8.quantize(self.x[k], self.fmt[k], self.rec, scale_in=self.scale[i:i + 1],
                                     amax_out=self.hist[i, 0:1])

    def update(self):
        fp8.fp8_update_amax_history(self.hist, self.scale, self.sinv, self.fmt_dev, len(self.names), self.L,
                                    self.algo, 0)


def checkpoint_roundtrip(tensors):
    """Save the delayed-scaling state to the host, lose the device copy, and
    restore it: the library keeps no state of its own, so the run must
    continue exactly as if nothing happened."""
    saved = [v.cpu().clone() for v in tensors]
    for v in tensors:
        v.fill_(float("nan"))
    for v, h in zip(tensors, saved):
        v.copy_(h.to(v.device))


def run_delayed(orc, base, fmts, algo, gemms, steps=50, full_steps=(0, 30, 49), gemm_steps=(0, 1, 30, 49),
                restore_at=25):
    L = 1024
    lay = DelayedLayer(base, fmts, L, algo)
    n = len(lay.names)
    hist_o = np.zeros((n, L), np.float32)
    scale_o = np.ones(n, np.float32)
    sinv_o = np.ones(n, np.float32)
    fmt_np = np.array([fmts[k] for k in lay.names], np.uint8)
    g = torch.Generator().manual_seed(77)
    for t in range(steps):
        lay.step_quantize(t)
        sync_ok()
        for i, k in enumerate(lay.names):
            f = fmts[k]
            xc = lay.x[k].cpu()
            xb = bits(xc)
            am = orc.amax_bf16(xb)
            hist_o[i, 0] = am if np.isnan(am) or np.isnan(hist_o[i, 0]) else max(hist_o[i, 0], am)
            q = lay.q[k]
            R, Cn = xc.shape
            # every byte of the first tensor at selected steps, sampled rows / columns otherwise
            if i == 0 and t in full_steps:
                ref = orc.quantize(xb, f, orc.DELAYED, scale_in=scale_o[i], amax_io=np.float32(0))
                assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], f, f"{k} t{t} row")
                assert_codes_equal(q.q_colT.cpu().numpy()[:, :R], ref["q_colT"], f, f"{k} t{t} colT")
            rows = torch.randperm(R, generator=g)[:4].numpy()
            cols = torch.randperm(Cn, generator=g)[:4].numpy()
            got_r = q.q_row[torch.from_numpy(rows).to(DEV)].cpu().numpy()
            exp_r = orc.cast_points(xb[rows], scale_o[i], f).reshape(len(rows), Cn)
            assert_codes_equal(got_r, exp_r, f, f"{k} t{t} rows")
            got_c = q.q_colT[torch.from_numpy(cols).to(DEV), :R].cpu().numpy()
            exp_c = orc.cast_points(np.ascontiguousarray(xb[:, cols].T), scale_o[i], f).reshape(len(cols), R)
            assert_codes_equal(got_c, exp_c, f, f"{k} t{t} cols")
            assert_f32_bits_equal(q.scale_inv_row.cpu().numpy(), np.array([np.float32(1) / scale_o[i]]),
                                  f"{k} t{t} sinv")
        assert_f32_bits_equal(lay.hist[:, 0].cpu().numpy(), hist_o[:, 0], f"amax t{t}")
        if t in gemm_steps:
            for gi, (a, al, b, bl) in enumerate(gemms):
                qa, qb = lay.q[a], lay.q[b]
                A = qa.q_row if al == "row" else qa.q_colT
                B = qb.q_row if bl == "row" else qb.q_colT
                K = lay.x[a].shape[1] if al == "row" else lay.x[a].shape[0]
                sa = qa.scale_inv_row if al == "row" else qa.scale_inv_col
                sb = qb.scale_inv_row if bl == "row" else qb.scale_inv_col
                C = fp8.scaled_gemm(A, fmts[a], B, fmts[b], sa, sb, K=K)
                sync_ok()
                sampled_gemm_check(orc, A[:, :K], fmts[a], B[:, :K], fmts[b], sa, sb, C, seed=t * 10 + gi,
                                   what=f"t{t} gemm {a}.{al} x {b}.{bl}", strict=True)
                del C
        lay.update()
        orc.update_amax_history(hist_o, scale_o, sinv_o, fmt_np, algo, 0)
        sync_ok()
        assert_f32_bits_equal(lay.hist.cpu().numpy(), hist_o, f"hist t{t}")
        assert_f32_bits_equal(lay.scale.cpu().numpy(), scale_o, f"scale t{t}")
        assert_f32_bits_equal(lay.sinv.cpu().numpy(), sinv_o, f"scale_inv t{t}")
        if t == restore_at:
            checkpoint_roundtrip((lay.hist, lay.scale, lay.sinv))
            sync_ok()
    # the spike at t = 30 must have lowered the activation scales afterwards
    return scale_o


MLP_GEMMS = [("x", "row", "w_gate", "row"), ("x", "row", "w_up", "row"), ("h", "row", "w_down", "row"),
             ("dy_down", "row", "w_down", "colT"), ("dy_gate", "row", "w_gate", "colT"),
             ("dy_up", "row", "w_up", "colT"), ("dy_down", "colT", "h", "colT"),
             ("dy_gate", "colT", "x", "colT"), ("dy_up", "colT", "x", "colT")]


def test_config2_llama_mlp_delayed_50_steps(orc):
    base = synth.llama_mlp_base()
    fmts = {k: (1 if k.startswith("dy") else 0) for k in base}          # hybrid: E5M2 gradients
    run_delayed(orc, base, fmts, orc.MOST_RECENT, MLP_GEMMS)


FLUX_GEMMS = [("x", "row", "w_qkv", "row"), ("x", "row", "w_up", "row"), ("h", "row", "w_down", "row"),
              ("dy_qkv", "row", "w_qkv", "colT"), ("dy_up", "row", "w_up", "colT"),
              ("dy_down", "row", "w_down", "colT"), ("dy_qkv", "colT", "x", "colT"),
              ("dy_up", "colT", "x", "colT"), ("dy_down", "colT", "h", "colT")]


def test_config5_flux_delayed_max_50_steps(orc):
    base = synth.flux_base()
    fmts = {k: 0 for k in base}                                         # all E4M3
    run_delayed(orc, base, fmts, orc.MAX, FLUX_GEMMS)


# --------------------------------------------------------------------------------------------
# 3. rowwise attention projections
# --------------------------------------------------------------------------------------------

def rowwise_layer_check(orc, t, fmts, gemms, seed):
    """Quantize every tensor with the rowwise recipe; check sampled rows and
    columns (bytes and scale_inv) against the oracle, then every GEMM on
    sampled rows, columns and points."""
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    q = {k: fp8.quantize(t[k].to(DEV), fmts[k], rec) for k in fmts}
    sync_ok()
    g = torch.Generator().manual_seed(seed)
    for k, f in fmts.items():
        xb = bits(t[k])
        R, Cn = xb.shape
        for r in torch.randperm(R, generator=g)[:8].tolist():
            ref = orc.quantize(xb[r:r + 1], f, orc.ROWWISE, layouts=1)
            assert_codes_equal(q[k].q_row[r:r + 1].cpu().numpy(), ref["q_row"], f, f"{k} row {r}")
            assert_f32_bits_equal(q[k].scale_inv_row[r:r + 1].cpu().numpy(), ref["scale_inv_row"], k)
        for c in torch.randperm(Cn, generator=g)[:8].tolist():
            ref = orc.quantize(np.ascontiguousarray(xb[:, c:c + 1]), f, orc.ROWWISE, layouts=2)
            assert_codes_equal(q[k].q_colT[c:c + 1, :R].cpu().numpy(), ref["q_colT"], f, f"{k} col {c}")
            assert_f32_bits_equal(q[k].scale_inv_col[c:c + 1].cpu().numpy(), ref["scale_inv_col"], k)
    for gi, (a, al, b, bl) in enumerate(gemms):
        A = q[a].q_row if al == "row" else q[a].q_colT
        B = q[b].q_row if bl == "row" else q[b].q_colT
        K = t[a].shape[1] if al == "row" else t[a].shape[0]
        sa = q[a].scale_inv_row if al == "row" else q[a].scale_inv_col
        sb = q[b].scale_inv_row if bl == "row" else q[b].scale_inv_col
        C = fp8.scaled_gemm(A, fmts[a], B, fmts[b], sa, sb, K=K)
        sync_ok()
        sampled_gemm_check(orc, A[:, :K], fmts[a], B[:, :K], fmts[b], sa, sb, C, seed=seed + gi,
                           what=f"{a}.{al} x {b}.{bl}")
        del C
    return q


def test_config3_llama_attention_rowwise(orc):
    """Config 3, attention projections: QKV and O under the rowwise recipe
    (Student-t activations), all six GEMMs; X's bytes and scales in full."""
    t = synth.llama_attn_extra()
    fmts = {"x": 0, "w_qkv": 0, "o_in": 0, "w_o": 0, "dy_qkv": 1, "dy_o": 1}
    gemms = [("x", "row", "w_qkv", "row"), ("o_in", "row", "w_o", "row"), ("dy_qkv", "row", "w_qkv", "colT"),
             ("dy_o", "row", "w_o", "colT"), ("dy_qkv", "colT", "x", "colT"), ("dy_o", "colT", "o_in", "colT")]
    q = rowwise_layer_check(orc, t, fmts, gemms, seed=5)
    xb = bits(t["x"])
    ref = orc.quantize(xb, 0, orc.ROWWISE)
    R = xb.shape[0]
    assert_codes_equal(q["x"].q_row.cpu().numpy(), ref["q_row"], 0, "x")
    assert_codes_equal(q["x"].q_colT.cpu().numpy()[:, :R], ref["q_colT"], 0, "x")
    assert_f32_bits_equal(q["x"].scale_inv_row.cpu().numpy(), ref["scale_inv_row"], "x")
    assert_f32_bits_equal(q["x"].scale_inv_col.cpu().numpy(), ref["scale_inv_col"], "x")


def test_config3_llama_mlp_rowwise(orc):
    """Config 3, MLP: gate, up and down under the rowwise recipe with
    Student-t activations, the nine GEMMs (fprop, dgrad, wgrad of each)."""
    t = synth.llama_rowwise_mlp()
    fmts = {k: (1 if k.startswith("dy") else 0) for k in t}
    rowwise_layer_check(orc, t, fmts, [g for g in MLP_GEMMS], seed=50)


# --------------------------------------------------------------------------------------------
# 4. DeepSeek-V3 MoE layer
# --------------------------------------------------------------------------------------------

def test_config4_moe_layer(orc):
    from test_gpu_gemm import offsets_of
    H, F, E = synth.DSV3["H"], synth.DSV3["F"], synth.DSV3["E"]
    sizes = synth.moe_group_sizes().numpy()
    assert (sizes == 0).sum() >= 8 and sizes.sum() == 32768
    off = offsets_of(sizes)
    off_d = torch.from_numpy(off).to(DEV)
    Mt = int(off[-1])
    tok = synth.moe_tokens()
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    # token side: rowwise + per-group colwise
    tf = {"xp": 0, "hp": 0, "dy_down": 1, "dy_gate": 1, "dy_up": 1}
    qt = {k: fp8.quantize(tok[k].to(DEV), f, rec, group_offsets=off_d, host_offsets=off) for k, f in tf.items()}
    # weights: rowwise per expert row, per-expert colwise (equal groups of `rows per expert`)
    w = {"w_gate": synth.moe_weight((E * F, H), DEV, seed=10), "w_up": synth.moe_weight((E * F, H), DEV, seed=12),
         "w_down": synth.moe_weight((E * H, F), DEV, seed=11)}
    woff = {"w_gate": np.arange(E + 1, dtype=np.int32) * F, "w_up": np.arange(E + 1, dtype=np.int32) * F,
            "w_down": np.arange(E + 1, dtype=np.int32) * H}
    qw = {k: fp8.quantize(w[k], 0, rec, group_offsets=torch.from_numpy(woff[k]).to(DEV), host_offsets=woff[k])
          for k in w}
    sync_ok()

    nz = np.nonzero(sizes)[0]
    g = torch.Generator().manual_seed(4)
    experts = {int(np.argmax(sizes)), int(nz[np.argmin(sizes[nz])])}
    experts |= set(int(e) for e in np.nonzero(sizes == 0)[0])
    experts |= set(torch.randint(0, E, (8,), generator=g).tolist())
    poff = orc.padded_offsets(off)

    # token-side bytes for the sampled experts (rows and a block of columns)
    for k, f in tf.items():
        xb = bits(tok[k])
        Cn = xb.shape[1]
        sc = qt[k].scale_inv_col.view(E, Cn)
        for e in sorted(experts):
            r0, r1 = off[e], off[e + 1]
            if r1 == r0:
                assert torch.all(sc[e] == 1.0)
                continue
            ref = orc.quantize(xb[r0:r1, :64], f, orc.ROWWISE, layouts=2)
            seg = qt[k].q_colT[:64, poff[e]:poff[e + 1]].cpu().numpy()
            assert_codes_equal(seg[:, :r1 - r0], ref["q_colT"], f, f"{k} expert {e}")
            assert not seg[:, r1 - r0:].any()
            assert_f32_bits_equal(sc[e, :64].cpu().numpy(), ref["scale_inv_col"], f"{k} scol {e}")
            rr = orc.quantize(xb[r0:min(r1, r0 + 4)], f, orc.ROWWISE, layouts=1)
            assert_codes_equal(qt[k].q_row[r0:min(r1, r0 + 4)].cpu().numpy(), rr["q_row"], f, f"{k} rows {e}")
    # weight bytes for the sampled experts
    for k in w:
        rows_e = H if k == "w_down" else F
        for e in sorted(experts)[:6]:
            wb = bits(w[k][e * rows_e:(e + 1) * rows_e].cpu())
            ref = orc.quantize(wb, 0, orc.ROWWISE)
            assert_codes_equal(qw[k].q_row[e * rows_e:(e + 1) * rows_e].cpu().numpy(), ref["q_row"], 0, f"{k} {e}")
            seg = qw[k].q_colT[:, e * rows_e:(e + 1) * rows_e].cpu().numpy()
            assert_codes_equal(seg, ref["q_colT"], 0, f"{k} colT {e}")

    # the nine grouped GEMMs: fprop gate / up / down (M), dgrad gate / up / down (M on the weights' transposed
    # layout), wgrad gate / up / down (K)
    Cg = fp8.grouped_gemm(fp8.GROUPED_M, qt["xp"].q_row, 0, qw["w_gate"].q_row, 0, off_d, Mt, F, H,
                          qt["xp"].scale_inv_row, qw["w_gate"].scale_inv_row)
    Cu = fp8.grouped_gemm(fp8.GROUPED_M, qt["xp"].q_row, 0, qw["w_up"].q_row, 0, off_d, Mt, F, H,
                          qt["xp"].scale_inv_row, qw["w_up"].scale_inv_row)
    dXu = fp8.grouped_gemm(fp8.GROUPED_M_BT, qt["dy_up"].q_row, 1, qw["w_up"].q_colT, 0, off_d, Mt, H, F,
                           qt["dy_up"].scale_inv_row, qw["w_up"].scale_inv_col, ld_T=qw["w_up"].ld_colT)
    Cd = fp8.grouped_gemm(fp8.GROUPED_M, qt["hp"].q_row, 0, qw["w_down"].q_row, 0, off_d, Mt, H, F,
                          qt["hp"].scale_inv_row, qw["w_down"].scale_inv_row)
    dX = fp8.grouped_gemm(fp8.GROUPED_M_BT, qt["dy_gate"].q_row, 1, qw["w_gate"].q_colT, 0, off_d, Mt, H, F,
                          qt["dy_gate"].scale_inv_row, qw["w_gate"].scale_inv_col, ld_T=qw["w_gate"].ld_colT)
    dH = fp8.grouped_gemm(fp8.GROUPED_M_BT, qt["dy_down"].q_row, 1, qw["w_down"].q_colT, 0, off_d, Mt, F, H,
                          qt["dy_down"].scale_inv_row, qw["w_down"].scale_inv_col, ld_T=qw["w_down"].ld_colT)
    dWg = fp8.grouped_gemm(fp8.GROUPED_K, qt["dy_gate"].q_colT, 1, qt["xp"].q_colT, 0, off_d, Mt, F, H,
                           qt["dy_gate"].scale_inv_col, qt["xp"].scale_inv_col, ld_T=qt["xp"].ld_colT)
    dWu = fp8.grouped_gemm(fp8.GROUPED_K, qt["dy_up"].q_colT, 1, qt["xp"].q_colT, 0, off_d, Mt, F, H,
                           qt["dy_up"].scale_inv_col, qt["xp"].scale_inv_col, ld_T=qt["xp"].ld_colT)
    dWd = fp8.grouped_gemm(fp8.GROUPED_K, qt["dy_down"].q_colT, 1, qt["hp"].q_colT, 0, off_d, Mt, H, F,
                           qt["dy_down"].scale_inv_col, qt["hp"].scale_inv_col, ld_T=qt["hp"].ld_colT)
    sync_ok()

    def cpu(t):
        return t.cpu().numpy()

    checks = [  # (output, A rows source, B expert matrix source, ...)
        ("fprop gate", Cg, qt["xp"], 0, lambda e: cpu(qw["w_gate"].q_row[e * F:(e + 1) * F]),
         lambda e: cpu(qw["w_gate"].scale_inv_row[e * F:(e + 1) * F]), 0, F),
        ("fprop up", Cu, qt["xp"], 0, lambda e: cpu(qw["w_up"].q_row[e * F:(e + 1) * F]),
         lambda e: cpu(qw["w_up"].scale_inv_row[e * F:(e + 1) * F]), 0, F),
        ("dgrad up", dXu, qt["dy_up"], 1, lambda e: cpu(qw["w_up"].q_colT[:, e * F:(e + 1) * F]),
         lambda e: cpu(qw["w_up"].scale_inv_col.view(E, H)[e]), 0, H),
        ("fprop down", Cd, qt["hp"], 0, lambda e: cpu(qw["w_down"].q_row[e * H:(e + 1) * H]),
         lambda e: cpu(qw["w_down"].scale_inv_row[e * H:(e + 1) * H]), 0, H),
        ("dgrad gate", dX, qt["dy_gate"], 1, lambda e: cpu(qw["w_gate"].q_colT[:, e * F:(e + 1) * F]),
         lambda e: cpu(qw["w_gate"].scale_inv_col.view(E, H)[e]), 0, H),
        ("dgrad down", dH, qt["dy_down"], 1, lambda e: cpu(qw["w_down"].q_colT[:, e * H:(e + 1) * H]),
         lambda e: cpu(qw["w_down"].scale_inv_col.view(E, F)[e]), 0, F),
    ]
    for name, C, qa, fa, Bexp, sbexp, fb, N in checks:
        Arow = qa.q_row
        for e in sorted(experts):
            r0, r1 = int(off[e]), int(off[e + 1])
            if r1 == r0:
                continue
            rows = np.arange(r0, r1)[torch.randperm(r1 - r0, generator=g)[:4].numpy()]
            pm = np.repeat(rows - r0, N).astype(np.int64)
            pn = np.tile(np.arange(N), len(rows)).astype(np.int64)
            ref, bound = orc.gemm(cpu(Arow[r0:r1]), fa, Bexp(e), fb, cpu(qa.scale_inv_row[r0:r1]), sbexp(e),
                                  points=(pm, pn))
            out = C[torch.from_numpy(pm + r0).to(DEV), torch.from_numpy(pn).to(DEV)].float().cpu().numpy()
            check_gemm(out, ref, bound, f"{name} expert {e}", strict=True)
    # wgrad of gate, up and down: dW_e = dY_e^T X_e over the group's rows
    for name, dW, qa, qb, Nw, Kw in (("wgrad gate", dWg, qt["dy_gate"], qt["xp"], F, H),
                                     ("wgrad up", dWu, qt["dy_up"], qt["xp"], F, H),
                                     ("wgrad down", dWd, qt["dy_down"], qt["hp"], H, F)):
        sca = qa.scale_inv_col.view(E, Nw)
        scb = qb.scale_inv_col.view(E, Kw)
        for e in sorted(experts):
            if sizes[e] == 0:
                assert torch.all(dW[e] == 0), f"{name} expert {e}"
                continue
            a = cpu(qa.q_colT[:, poff[e]:poff[e] + sizes[e]])
            b = cpu(qb.q_colT[:, poff[e]:poff[e] + sizes[e]])
            rows = torch.randperm(Nw, generator=g)[:4].numpy()
            pm = np.repeat(rows, Kw).astype(np.int64)
            pn = np.tile(np.arange(Kw), len(rows)).astype(np.int64)
            ref, bound = orc.gemm(a, 1, b, 0, cpu(sca[e]), cpu(scb[e]), points=(pm, pn))
            out = dW[e][torch.from_numpy(pm).to(DEV), torch.from_numpy(pn).to(DEV)].float().cpu().numpy()
            check_gemm(out, ref, bound, f"{name} expert {e}")
    ldT = qt["xp"].ld_colT
    assert ldT >= int(poff[-1])
