"""Benchmark of the FP8 linear hot path on one GB300 (or N, one process each).

Default workload (`--workload llama_mlp`): one step = the whole FP8 path of
the Llama-3-8B MLP block (tokens 8192, hidden 4096, ffn 14336) under delayed
scaling with the hybrid format:
  8 fused quantizes (X, W_gate, W_up, W_down, H, dY_down, dY_gate, dY_up;
    E4M3 forward / E5M2 gradients; rowwise + colwise-transposed layouts),
  9 FP8 GEMMs (fprop, dgrad, wgrad of gate, up and down; 962 GFLOP each),
  1 fused amax-history update (8 histories of length 1024, most_recent).
Under torchrun each rank runs its own batch (data parallel, weak scaling);
the one exchange of the path -- a MAX all-reduce of the current amaxes before
the update -- goes over NCCL.

Other workloads (same JSON line, their own config):
  llama_rowwise  Llama-3-8B attention projections + MLP, rowwise recipe,
                 Student-t activations (15 GEMMs, 11.13 TFLOP per step)
  moe            DeepSeek-V3-shaped MoE layer: 32768 routed rows, 256 experts,
                 hidden 7168, ffn 2048; rowwise tokens with per-expert colwise
                 scales, rowwise / per-expert colwise weights; the routed rows
                 gathered and SwiGLU applied inside their quantizes; gate|up
                 fused: 6 grouped GEMMs with the FLOPs of 9
  moe_unfused    the same layer with the routed rows and the down projection's
                 input given as bf16 tensors, separate gate and up (9 GEMMs)
  flux           Flux-12B linears (tokens 9216, hidden 3072, MLP 12288, QKV
                 9216), delayed scaling, all E4M3, amax algo max
  llama_mxfp8    the Llama-3-8B MLP step under the MXFP8 recipe (blocks of 32
                 with E8M0 scales, both layouts per tensor, block-scaled GEMMs)
  moe_mxfp8      the DeepSeek-V3 MoE layer under the MXFP8 recipe with the
                 fused permute / SwiGLU prologues and MX grouped GEMMs
  llama_blockwise  the same step under the blockwise recipe (1x128 activation
                 and gradient blocks, 128x128 weight blocks, power-of-two scales)
  bw_quantize    the blockwise quantize of dY_gate (1x128 blocks)
  rowwise_quantize  the rowwise (current scaling) quantize of dY_gate
  rowwise_resident  the single-launch rowwise quantize of X [8192, 4096],
                 also timed against the two-pass path
  sweep          the delayed quantize (E4M3, both layouts) of 2^20 .. 2^30
                 elements, GB/s against size
  gemm, quantize single kernels of the default step, for profiling
  grouped_m, grouped_k  one M-grouped / K-grouped expert GEMM of a reduced
                 MoE layer (64 experts, 8192 routed rows), for profiling
  mx_grouped_m, mx_grouped_k  the MXFP8 M-grouped fprop / K-grouped wgrad of
                 that layer, for profiling
  quantize_grouped  the rowwise quantize of one reduced MoE weight (64
                 experts x 2048 rows x 7168), for profiling
  stack_quantize, mx_stack_quantize  the rowwise (256 equal groups) / MX
                 quantize of a whole DeepSeek-V3 expert-weight stack, as the
                 MoE steps run it: gate|up [256 x 4096, 7168], or with
                 --stack down [256 x 7168, 2048]
  mx_gemm, mx_quantize  the MXFP8 gate GEMM / the MX quantize of dY_gate
  mx_permute, mx_swiglu  fused MoE prologue + MX quantize at DeepSeek-V3
                 shapes (gather of 4096 x top-8 routed rows of 7168; SwiGLU
                 of [32768, 2 x 2048]), also timed against the unfused chain
  permute, swiglu  the same prologues fused into the rowwise quantize with
                 per-expert column scales, also timed against the unfused chain

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 linear fwd+bwd TFLOPS & quantize GB/s per GB300, as % of roofline"
L_HIST = 1024
QUANT_BYTES_PER_ELEM = 4                  # 2 B read + 1 B per layout, two layouts

# DRAM bytes (read + write) of one launch of the step's dominant kernel (the
# gate GEMM 8192x14336x4096) from one ncu capture; reported only while the
# sources it was taken on are unchanged (checked by hash).
GEMM_TRAFFIC = {
    "llama_mlp": {"bytes": 317.7e6, "kernel": "fp8_gemm_pair_kernel",
                  "sources": {"gemm.cu": "54081648946ce4ea", "fp8gb_device.cuh": "b07d3da7b8f74a94"}},
    # the blockwise step's dominant kernel is the same dense MX GEMM on the same shapes
    "llama_blockwise": {"bytes": 307.0e6, "kernel": "mx_gemm_kernel",
                        "sources": {"mxgemm.cu": "9045884819bbbe90", "fp8gb_device.cuh": "b07d3da7b8f74a94"}},
    "llama_mxfp8": {"bytes": 307.0e6, "kernel": "mx_gemm_kernel",
                    "sources": {"mxgemm.cu": "9045884819bbbe90", "fp8gb_device.cuh": "b07d3da7b8f74a94"}},
}


def gemm_traffic(name):
    import hashlib
    entry = GEMM_TRAFFIC.get(name)
    if entry is None:
        return None
    csrc = os.path.join(ROOT, "fp8_mixed_precision_scale_gb300", "csrc")
    for fname, want in entry["sources"].items():
        with open(os.path.join(csrc, fname), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != want:
                return None
    return entry["bytes"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms; only the
    samples taken inside the timed window are kept."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (host time, csv line)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if window is not None and not (window[0] <= ts <= window[1]):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------------------------

def _timed(ev, kind, fn, work=None):
    """Run fn; with ev, bracket it with CUDA events on the current stream and
    record (start, end, work) under `kind`."""
    if ev is None:
        fn()
        return
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    ev.setdefault(kind, []).append((a, b, work))


def _normal(g, dev, shape, std):
    return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)


def quantize_bytes(shape, layouts=3):
    """Algorithmic bytes of one quantize: 2 B read + 1 B per emitted layout per element."""
    r, c = shape
    return r * c * (2 + (1 if layouts & 1 else 0) + (1 if layouts & 2 else 0))


class DelayedStep:
    """A block of Linears under delayed scaling: quantize (stored scale,
    amax into the history slot), GEMMs with per-tensor scales, one update."""

    def __init__(self, dev, seed, shapes, fmts, gemms, fwd_q, bwd_q, n_fwd_gemm, algo, tokens, name, desc,
                 keys=None, outs=None):
        import fp8_mixed_precision_scale_gb300 as fp8
        self.fp8 = fp8
        self.name, self.desc, self.tokens, self.algo = name, desc, tokens, algo
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.order = list(shapes)
        self.inp = {k: _normal(g, dev, *shapes[k]) for k in self.order if keys is None or k in keys}
        self.fmt = fmts
        self.gemms, self.fwd_q, self.bwd_q, self.n_fwd_gemm = gemms, fwd_q, bwd_q, n_fwd_gemm
        n = len(self.order)
        self.hist = torch.zeros((n, L_HIST), dtype=torch.float32, device=dev)
        self.scale = torch.ones(n, dtype=torch.float32, device=dev)
        self.scale_inv = torch.ones(n, dtype=torch.float32, device=dev)
        self.fmt_dev = torch.tensor([fmts[k] for k in self.order], dtype=torch.uint8, device=dev)
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, r), dtype=torch.uint8, device=dev),
                             srow=torch.empty(1, dtype=torch.float32, device=dev),
                             scol=torch.empty(1, dtype=torch.float32, device=dev))
        self.out, self.gemm_work = {}, {}
        self.flops = 0.0
        for (a, al, b, bl, o) in gemms:
            M, K = shapes[a][0] if al == "row" else shapes[a][0][::-1]
            N = shapes[b][0][0] if bl == "row" else shapes[b][0][1]
            self.gemm_work[o] = (2.0 * M * N * K, M * K + N * K + 2.0 * M * N)
            self.flops += 2.0 * M * N * K
            if outs is None or o in outs:
                self.out[o] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.recipe = fp8.Recipe(kind=fp8.DELAYED, margin=0, history_len=L_HIST, algo=algo)
        self.q_bytes = sum(quantize_bytes(shapes[k][0]) for k in self.order)
        self.launches_per_step = len(self.order) + len(gemms) + 1
        self.d2h = [self.out[gemms[self.n_fwd_gemm - 1][4]]] if outs is None else []

    def quantize(self, k):
        i = self.order.index(k)
        t, q = self.inp[k], self.q[k]
        r, c = t.shape
        self.fp8.fp8_quantize(t, r, c, c, self.fmt[k], self.recipe, 3, self.scale[i:i + 1],
                              self.hist[i, 0:1], q["row"], q["srow"], q["colT"], r, q["scol"])

    def gemm(self, a, a_layout, b, b_layout, out):
        qa, qb = self.q[a], self.q[b]
        A = qa["row"] if a_layout == "row" else qa["colT"]
        B = qb["row"] if b_layout == "row" else qb["colT"]
        sa = qa["srow"] if a_layout == "row" else qa["scol"]
        sb = qb["srow"] if b_layout == "row" else qb["scol"]
        C = self.out[out]
        M, K = A.shape
        N = B.shape[0]
        self.fp8.fp8_scaled_gemm(A, self.fmt[a], K, B, self.fmt[b], K, M, N, K, sa, 0, sb, 0, C, N)

    def run(self, ev=None, world=1):
        for k in self.fwd_q:
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        for g in self.gemms[:self.n_fwd_gemm]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])
        for k in self.bwd_q:
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        for g in self.gemms[self.n_fwd_gemm:]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])
        if world > 1:
            from fp8_mixed_precision_scale_gb300 import dp
            dp.reduce_current_amax(self.hist)
        _timed(ev, "u", lambda: self.fp8.fp8_update_amax_history(
            self.hist, self.scale, self.scale_inv, self.fmt_dev, len(self.order), L_HIST, self.algo, 0),
            len(self.order) * (8.0 * L_HIST + 8))


T_, H_, F_ = 8192, 4096, 14336
LLAMA_MLP_SHAPES = {"x": ((T_, H_), 1.0), "w_gate": ((F_, H_), 0.02), "w_up": ((F_, H_), 0.02),
                    "w_down": ((H_, F_), 0.02), "h": ((T_, F_), 1.0), "dy_down": ((T_, H_), 1e-4),
                    "dy_gate": ((T_, F_), 1e-4), "dy_up": ((T_, F_), 1e-4)}
MLP_GEMMS = [  # (A, A layout, B, B layout, output)
    ("x", "row", "w_gate", "row", "gate"),             # fprop gate
    ("x", "row", "w_up", "row", "up"),                 # fprop up
    ("h", "row", "w_down", "row", "y"),                # fprop down
    ("dy_down", "row", "w_down", "colT", "dh"),        # dgrad down
    ("dy_gate", "row", "w_gate", "colT", "dx_gate"),   # dgrad gate
    ("dy_up", "row", "w_up", "colT", "dx_up"),         # dgrad up
    ("dy_down", "colT", "h", "colT", "dw_down"),       # wgrad down
    ("dy_gate", "colT", "x", "colT", "dw_gate"),       # wgrad gate
    ("dy_up", "colT", "x", "colT", "dw_up"),           # wgrad up
]
LLAMA_MLP_DESC = ("llama3-8b-mlp fwd+bwd, delayed scaling: tokens 8192, hidden 4096, ffn 14336, "
                  "hybrid e4m3 fwd / e5m2 grads, amax history 1024 most_recent, margin 0")


def llama_mlp_step(dev, seed, keys=None, outs=None):
    import fp8_mixed_precision_scale_gb300 as fp8
    fmts = {k: (fp8.E5M2 if k.startswith("dy") else fp8.E4M3FN) for k in LLAMA_MLP_SHAPES}
    return DelayedStep(dev, seed, LLAMA_MLP_SHAPES, fmts, MLP_GEMMS, ["x", "w_gate", "w_up", "w_down", "h"],
                       ["dy_down", "dy_gate", "dy_up"], 3, fp8.MOST_RECENT, T_, "llama_mlp", LLAMA_MLP_DESC,
                       keys, outs)


FT, FH, FF, FQ = 9216, 3072, 12288, 9216
FLUX_SHAPES = {"x": ((FT, FH), 1.0), "w_qkv": ((FQ, FH), 0.02), "w_up": ((FF, FH), 0.02),
               "w_down": ((FH, FF), 0.02), "h": ((FT, FF), 1.0), "dy_qkv": ((FT, FQ), 1e-4),
               "dy_up": ((FT, FF), 1e-4), "dy_down": ((FT, FH), 1e-4)}
FLUX_GEMMS = [("x", "row", "w_qkv", "row", "qkv"), ("x", "row", "w_up", "row", "up"),
              ("h", "row", "w_down", "row", "y"), ("dy_qkv", "row", "w_qkv", "colT", "dx_qkv"),
              ("dy_up", "row", "w_up", "colT", "dx_up"), ("dy_down", "row", "w_down", "colT", "dh"),
              ("dy_qkv", "colT", "x", "colT", "dw_qkv"), ("dy_up", "colT", "x", "colT", "dw_up"),
              ("dy_down", "colT", "h", "colT", "dw_down")]


def flux_step(dev, seed):
    import fp8_mixed_precision_scale_gb300 as fp8
    fmts = {k: fp8.E4M3FN for k in FLUX_SHAPES}
    desc = ("flux-12b linears fwd+bwd (QKV 3072->9216, MLP 3072->12288->3072), tokens 2 x (4096 + 512) = 9216, "
            "delayed scaling, all e4m3, amax history 1024, algo max, margin 0")
    return DelayedStep(dev, seed, FLUX_SHAPES, fmts, FLUX_GEMMS, ["x", "w_qkv", "w_up", "w_down", "h"],
                       ["dy_qkv", "dy_up", "dy_down"], 3, fp8.MAX, FT, "flux", desc)


class RowwiseStep:
    """Llama-3-8B attention projections + MLP with the rowwise recipe: every
    tensor quantized with per-row scales (row layout) and per-column scales
    (transposed layout); GEMMs with per-row / per-column scales."""

    SHAPES = {  # name: (shape, distribution, fmt)
        "x": ((T_, H_), "t", 0), "w_qkv": ((6144, H_), 0.02, 0), "o_in": ((T_, 6144), "t", 0),
        "w_o": ((H_, 6144), 0.02, 0), "x2": ((T_, H_), "t", 0), "w_gate": ((F_, H_), 0.02, 0),
        "w_up": ((F_, H_), 0.02, 0), "w_down": ((H_, F_), 0.02, 0), "h": ((T_, F_), "t", 0),
        "dy_qkv": ((T_, 6144), 1e-4, 1), "dy_o": ((T_, H_), 1e-4, 1), "dy_gate": ((T_, F_), 1e-4, 1),
        "dy_up": ((T_, F_), 1e-4, 1), "dy_down": ((T_, H_), 1e-4, 1)}
    GEMMS = [("x", "row", "w_qkv", "row", "qkv"), ("o_in", "row", "w_o", "row", "o"),
             ("x2", "row", "w_gate", "row", "gate"), ("x2", "row", "w_up", "row", "up"),
             ("h", "row", "w_down", "row", "y"),
             ("dy_down", "row", "w_down", "colT", "dh"), ("dy_gate", "row", "w_gate", "colT", "dx_gate"),
             ("dy_up", "row", "w_up", "colT", "dx_up"), ("dy_o", "row", "w_o", "colT", "do_in"),
             ("dy_qkv", "row", "w_qkv", "colT", "dx"),
             ("dy_down", "colT", "h", "colT", "dw_down"), ("dy_gate", "colT", "x2", "colT", "dw_gate"),
             ("dy_up", "colT", "x2", "colT", "dw_up"), ("dy_o", "colT", "o_in", "colT", "dw_o"),
             ("dy_qkv", "colT", "x", "colT", "dw_qkv")]
    FWD_Q = ["x", "w_qkv", "o_in", "w_o", "x2", "w_gate", "w_up", "w_down", "h"]
    BWD_Q = ["dy_down", "dy_gate", "dy_up", "dy_o", "dy_qkv"]

    def __init__(self, dev, seed, keys=None):
        import fp8_mixed_precision_scale_gb300 as fp8
        import synth
        self.fp8 = fp8
        self.name = "llama_rowwise"
        self.desc = ("llama3-8b attention projections (QKV 4096->6144, O 6144->4096) + MLP (4096->14336->4096) "
                     "fwd+bwd, rowwise recipe: per-row scales for the row layout, per-column scales for the "
                     "transposed layout; tokens 8192; Student-t (nu=4) activations; hybrid e4m3 / e5m2")
        self.tokens = T_
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.inp, self.fmt = {}, {}
        for k, (shape, dist, f) in self.SHAPES.items():
            if keys is not None and k not in keys:
                continue
            self.inp[k] = synth.student_t(shape, 4, g, dev) if dist == "t" else _normal(g, dev, shape, dist)
            self.fmt[k] = f
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, r), dtype=torch.uint8, device=dev),
                             srow=torch.empty(r, dtype=torch.float32, device=dev),
                             scol=torch.empty(c, dtype=torch.float32, device=dev))
        self.out, self.gemm_work = {}, {}
        self.flops = 0.0
        for (a, al, b, bl, o) in self.GEMMS:
            if a not in self.inp or b not in self.inp:
                continue
            M, K = self.inp[a].shape if al == "row" else self.inp[a].shape[::-1]
            N = self.inp[b].shape[0] if bl == "row" else self.inp[b].shape[1]
            self.out[o] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.gemm_work[o] = (2.0 * M * N * K, M * K + N * K + 2.0 * M * N)
            self.flops += 2.0 * M * N * K
        self.recipe = fp8.Recipe(kind=fp8.ROWWISE)
        self.q_bytes = sum(quantize_bytes(t.shape) for t in self.inp.values())
        self.launches_per_step = 4 * len(self.inp) + len(self.GEMMS)   # clear, amax, cast, finalise per tensor
        self.d2h = [self.out["y"]] if "y" in self.out else []

    def quantize(self, k):
        t, q = self.inp[k], self.q[k]
        r, c = t.shape
        self.fp8.fp8_quantize(t, r, c, c, self.fmt[k], self.recipe, 3, None, None, q["row"], q["srow"],
                              q["colT"], r, q["scol"])

    def quantize_resident(self, k):
        """The same quantize through the single-launch entry point."""
        t, q = self.inp[k], self.q[k]
        r, c = t.shape
        self.fp8.fp8_quantize_rowwise_resident(t, r, c, c, self.fmt[k], 0, 3, None, q["row"], q["srow"],
                                               q["colT"], r, q["scol"])

    def gemm(self, a, al, b, bl, out):
        qa, qb = self.q[a], self.q[b]
        A = qa["row"] if al == "row" else qa["colT"]
        B = qb["row"] if bl == "row" else qb["colT"]
        sa = qa["srow"] if al == "row" else qa["scol"]
        sb = qb["srow"] if bl == "row" else qb["scol"]
        M, K = A.shape
        N = B.shape[0]
        self.fp8.fp8_scaled_gemm(A, self.fmt[a], K, B, self.fmt[b], K, M, N, K, sa, 1, sb, 1, self.out[out], N)

    def run(self, ev=None, world=1):
        for k in self.FWD_Q:
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        for g in self.GEMMS[:5]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])
        for k in self.BWD_Q:
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        for g in self.GEMMS[5:]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])


class TinyStep(RowwiseStep):
    """The tiny FP8 linear of the benchmark set (its inputs from synth.tiny):
    X [256, 512] ~ N(0, 1) with 0.1 % of the entries x50, W [512, 512] ~ N(0,
    0.02), dY [256, 512] ~ N(0, 1e-3); rowwise recipe, X and W in e4m3, dY in
    e5m2; fprop, dgrad and wgrad GEMMs.  Launch-bound: its inputs sit in L2."""

    GEMMS = [("x", "row", "w", "row", "y"), ("dy", "row", "w", "colT", "dx"), ("dy", "colT", "x", "colT", "dw")]

    def __init__(self, dev, seed, keys=None):
        import fp8_mixed_precision_scale_gb300 as fp8
        import synth
        self.fp8 = fp8
        self.name = "tiny"
        self.desc = ("tiny fp8 linear fwd+bwd: X [256,512] N(0,1) with 0.1% entries x50, W [512,512] N(0,0.02), "
                     "dY [256,512] N(0,1e-3); rowwise recipe, e4m3 X/W, e5m2 dY")
        self.tokens = 256
        self.inp = {k: v.to(dev) for k, v in synth.tiny().items()}
        self.fmt = {"x": 0, "w": 0, "dy": 1}
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, r), dtype=torch.uint8, device=dev),
                             srow=torch.empty(r, dtype=torch.float32, device=dev),
                             scol=torch.empty(c, dtype=torch.float32, device=dev))
        self.out, self.gemm_work = {}, {}
        self.flops = 0.0
        for (a, al, b, bl, o) in self.GEMMS:
            M, K = self.inp[a].shape if al == "row" else self.inp[a].shape[::-1]
            N = self.inp[b].shape[0] if bl == "row" else self.inp[b].shape[1]
            self.out[o] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.gemm_work[o] = (2.0 * M * N * K, M * K + N * K + 2.0 * M * N)
            self.flops += 2.0 * M * N * K
        self.recipe = fp8.Recipe(kind=fp8.ROWWISE)
        self.q_bytes = sum(quantize_bytes(t.shape) for t in self.inp.values())
        self.launches_per_step = 4 * len(self.inp) + len(self.GEMMS)
        self.d2h = [self.out["y"]]

    def run(self, ev=None, world=1):
        for k in ("x", "w"):
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        _timed(ev, "g", lambda: self.gemm(*self.GEMMS[0]), self.gemm_work["y"])
        _timed(ev, "q", lambda: self.quantize("dy"), quantize_bytes(self.inp["dy"].shape))
        for g in self.GEMMS[1:]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])


def mx_quantize_bytes(shape):
    """Algorithmic bytes of one MX quantize with both layouts: 2 B read, 1 B
    per layout per element, one E8M0 byte per 32 elements per layout."""
    r, c = shape
    return r * c * 4 + 2 * (r * c // 32)


class MxStep:
    """The Llama-3-8B MLP block fwd+bwd under the MXFP8 recipe: every tensor
    MX-quantized once into both layouts (blocks of 32 along rows for the row
    layout, along columns for the transposed one, E8M0 scales); the nine
    GEMMs on the block-scaled tensor cores.  No history, no update."""

    def __init__(self, dev, seed, keys=None, outs=None, recipe="mxfp8"):
        import fp8_mixed_precision_scale_gb300 as fp8
        self.fp8 = fp8
        self.recipe = recipe
        self.name = "llama_" + recipe
        if recipe == "mxfp8":
            self.desc = ("llama3-8b-mlp fwd+bwd, mxfp8 recipe (OCP MX: 32-element blocks, E8M0 scales): tokens 8192, "
                         "hidden 4096, ffn 14336, e4m3 fwd / e5m2 grads")
        else:
            self.desc = ("llama3-8b-mlp fwd+bwd, blockwise recipe (1x128 activation / gradient blocks, 128x128 weight "
                         "blocks, power-of-two scales, block-scaled GEMMs): tokens 8192, hidden 4096, ffn 14336, "
                         "e4m3 fwd / e5m2 grads")
        self.tokens = T_
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.inp = {k: _normal(g, dev, *LLAMA_MLP_SHAPES[k]) for k in LLAMA_MLP_SHAPES if keys is None or k in keys}
        self.fmt = {k: (fp8.E5M2 if k.startswith("dy") else fp8.E4M3FN) for k in LLAMA_MLP_SHAPES}
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, r), dtype=torch.uint8, device=dev),
                             srow=torch.empty(fp8.fp8_mx_scale_bytes(r, c // 32), dtype=torch.uint8, device=dev),
                             scol=torch.empty(fp8.fp8_mx_scale_bytes(c, r // 32), dtype=torch.uint8, device=dev))
        self.out, self.gemm_work = {}, {}
        self.flops = 0.0
        for (a, al, b, bl, o) in MLP_GEMMS:
            M, K = LLAMA_MLP_SHAPES[a][0] if al == "row" else LLAMA_MLP_SHAPES[a][0][::-1]
            N = LLAMA_MLP_SHAPES[b][0][0] if bl == "row" else LLAMA_MLP_SHAPES[b][0][1]
            self.gemm_work[o] = (2.0 * M * N * K, M * K + N * K + 2.0 * M * N + (M + N) * K / 32)
            self.flops += 2.0 * M * N * K
            if outs is None or o in outs:
                self.out[o] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.q_bytes = sum(mx_quantize_bytes(LLAMA_MLP_SHAPES[k][0]) for k in LLAMA_MLP_SHAPES)
        self.launches_per_step = len(LLAMA_MLP_SHAPES) + len(MLP_GEMMS)
        self.d2h = [self.out["y"]] if outs is None else []

    def quantize(self, k):
        t, q = self.inp[k], self.q[k]
        r, c = t.shape
        if self.recipe == "blockwise":
            self.fp8.fp8_blockwise_quantize(t, r, c, c, self.fmt[k], 128 if k.startswith("w_") else 1, 3, q["row"],
                                            q["srow"], q["colT"], r, q["scol"])
        else:
            self.fp8.fp8_mx_quantize(t, r, c, c, self.fmt[k], 3, q["row"], q["srow"], q["colT"], r, q["scol"])

    def gemm(self, a, al, b, bl, out):
        qa, qb = self.q[a], self.q[b]
        A = qa["row"] if al == "row" else qa["colT"]
        B = qb["row"] if bl == "row" else qb["colT"]
        sA = qa["srow"] if al == "row" else qa["scol"]
        sB = qb["srow"] if bl == "row" else qb["scol"]
        M, K = A.shape
        N = B.shape[0]
        self.fp8.fp8_mx_gemm(A, self.fmt[a], K, sA, B, self.fmt[b], K, sB, M, N, K, self.out[out], N)

    def run(self, ev=None, world=1):
        for k in ["x", "w_gate", "w_up", "w_down", "h"]:
            _timed(ev, "q", lambda k=k: self.quantize(k), mx_quantize_bytes(self.inp[k].shape))
        for g in MLP_GEMMS[:3]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])
        for k in ["dy_down", "dy_gate", "dy_up"]:
            _timed(ev, "q", lambda k=k: self.quantize(k), mx_quantize_bytes(self.inp[k].shape))
        for g in MLP_GEMMS[3:]:
            _timed(ev, "g", lambda g=g: self.gemm(*g), self.gemm_work[g[4]])


class MoeStep:
    """DeepSeek-V3-shaped MoE layer fwd+bwd on one GPU under the rowwise
    recipe: rowwise scales per routed token row plus per-expert column
    scales, expert weights with per-row scales and per-expert column scales.
    The fused prologues do the token-side work in the quantizes: the routed
    rows are gathered from the 4096 token rows inside their quantize
    (fp8_permute_quantize), and SwiGLU of the fused gate|up projection's
    output is applied inside the quantize of the down projection's input
    (fp8_swiglu_quantize).  Gate and up are one [E, 2F, H] weight, so six
    grouped GEMMs carry the FLOPs of nine: M-grouped fprop (gate|up, down),
    M-grouped dgrad on the weights' transposed layouts, K-grouped wgrad."""

    def __init__(self, dev, seed):
        import numpy as np

        import fp8_mixed_precision_scale_gb300 as fp8
        import synth
        self.fp8 = fp8
        E, H, F, T = synth.DSV3["E"], synth.DSV3["H"], synth.DSV3["F"], synth.DSV3["tokens"]
        self.E, self.H, self.F = E, H, F
        sizes = synth.moe_group_sizes().numpy()
        self.sizes = sizes
        self.off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        self.off_h = torch.from_numpy(self.off)
        self.off_d = self.off_h.to(dev)
        self.M = M = int(self.off[-1])
        self.tokens = T
        self.name = "moe"
        self.desc = ("deepseek-v3 moe layer fwd+bwd, rowwise recipe: 4096 tokens x top-8 = 32768 routed rows gathered "
                     "into expert order inside their quantize, hidden 7168, 256 experts of ffn 2048 (gate|up fused, "
                     "down), SwiGLU fused into the quantize of the down projection's input, group sizes multinomial "
                     "over zipf(1.1) with 8 empty experts; rowwise + per-expert colwise scales; 6 grouped GEMMs (the "
                     "FLOPs of 9)")
        rng = np.random.default_rng(seed)
        self.src = torch.from_numpy(rng.integers(0, T, size=M).astype(np.int32)).to(dev)   # routed row -> token
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.inp = {"x": _normal(g, dev, (T, H), 1.0), "w_gu": _normal(g, dev, (E * 2 * F, H), 0.02),
                    "w_down": _normal(g, dev, (E * H, F), 0.02), "dy": _normal(g, dev, (M, H), 1e-4),
                    "dgu": _normal(g, dev, (M, 2 * F), 1e-4)}
        self.fmt = {"xp": 0, "hp": 0, "w_gu": 0, "w_down": 0, "dy": 1, "dgu": 1}
        self.recipe = fp8.Recipe(kind=fp8.ROWWISE)
        ldT = fp8.fp8_group_padded_offsets(self.off)[0]
        self.ldT_tok = max(16, (ldT + 15) // 16 * 16)
        self.q_shapes = {"xp": (M, H), "w_gu": (E * 2 * F, H), "w_down": (E * H, F), "hp": (M, F), "dy": (M, H),
                         "dgu": (M, 2 * F)}
        self.q = {}
        for k, (r, c) in self.q_shapes.items():
            ld = r if k.startswith("w_") else self.ldT_tok
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, ld), dtype=torch.uint8, device=dev), ldT=ld,
                             srow=torch.empty(r, dtype=torch.float32, device=dev),
                             scol=torch.empty(E * c, dtype=torch.float32, device=dev))
        e = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.out = {"gu": e(M, 2 * F), "y": e(M, H), "dh": e(M, F), "dx": e(M, H), "dw_down": e(E, H, F),
                    "dw_gu": e(E, 2 * F, H)}
        nz = int((sizes > 0).sum())
        fl = 2.0 * M * F * H
        self.gemm_work = {  # (flops, algorithmic bytes: A + non-empty experts' weights + C)
            "fprop_gu": (2 * fl, M * H + 2 * nz * F * H + 4.0 * M * F),
            "fprop_down": (fl, M * F + nz * F * H + 2.0 * M * H),
            "dgrad_down": (fl, M * H + nz * F * H + 2.0 * M * F),
            "dgrad_gu": (2 * fl, 2 * M * F + 2 * nz * F * H + 2.0 * M * H),
            "wgrad_down": (fl, M * (F + H) + 2.0 * E * F * H),
            "wgrad_gu": (2 * fl, M * (2 * F + H) + 4.0 * E * F * H)}
        self.flops = 9 * fl
        # algorithmic quantize bytes: 2 B read + 1 B per layout per element; SwiGLU reads gate and up
        self.q_work = {k: quantize_bytes(sh) + (2 * sh[0] * sh[1] if k == "hp" else 0)
                       for k, sh in self.q_shapes.items()}
        self.q_bytes = sum(self.q_work.values())
        # a grouped rowwise quantize is 5 launches (clear, amax, scales, cast, scales), an equal-groups one 4
        self.launches_per_step = 5 * 4 + 4 * 2 + 6
        self.d2h = [self.out["y"]]

    def quantize(self, k):
        fp8, q, E = self.fp8, self.q[k], self.E
        if k == "xp":
            x = self.inp["x"]
            fp8.fp8_permute_quantize(x, x.shape[0], x.shape[1], x.stride(0), self.src, self.M, 0, 0, 3, None,
                                     q["row"], q["srow"], q["colT"], q["ldT"], q["scol"], self.off_d, E)
        elif k == "hp":
            gu = self.out["gu"]
            fp8.fp8_swiglu_quantize(gu, self.M, self.F, gu.stride(0), 0, 0, 3, None, 0, None, q["row"], q["srow"],
                                    q["colT"], q["ldT"], q["scol"], self.off_d, E)
        else:
            t = self.inp[k]
            r, c = t.shape
            # expert weights: E equal groups (no offsets needed); routed tokens: the routing offsets
            off = None if k.startswith("w_") else self.off_d
            fp8.fp8_quantize(t, r, c, c, self.fmt[k], self.recipe, 3, None, None, q["row"], q["srow"], q["colT"],
                             q["ldT"], q["scol"], off, E)

    def run(self, ev=None, world=1):
        fp8, q, o, E, H, F, M = self.fp8, self.q, self.out, self.E, self.H, self.F, self.M
        GM, GK, GMT = fp8.GROUPED_M, fp8.GROUPED_K, fp8.GROUPED_M_BT
        off = self.off_d

        def gg(mode, a, al, b, bl, N, K, out, ldT=0):
            A = q[a]["row"] if al == "row" else q[a]["colT"]
            B = q[b]["row"] if bl == "row" else q[b]["colT"]
            sa = q[a]["srow"] if al == "row" else q[a]["scol"]
            sb = q[b]["srow"] if bl == "row" else q[b]["scol"]
            fp8.fp8_grouped_gemm(mode, A, self.fmt[a], B, self.fmt[b], off, E, M, N, K, sa, 1, sb, 1, o[out], ldT)

        W = self.gemm_work
        for k in ("xp", "w_gu", "w_down"):
            _timed(ev, "q", lambda k=k: self.quantize(k), self.q_work[k])
        _timed(ev, "g", lambda: gg(GM, "xp", "row", "w_gu", "row", 2 * F, H, "gu"), W["fprop_gu"])
        _timed(ev, "q", lambda: self.quantize("hp"), self.q_work["hp"])
        _timed(ev, "g", lambda: gg(GM, "hp", "row", "w_down", "row", H, F, "y"), W["fprop_down"])
        for k in ("dy", "dgu"):
            _timed(ev, "q", lambda k=k: self.quantize(k), self.q_work[k])
        _timed(ev, "g", lambda: gg(GMT, "dy", "row", "w_down", "colT", F, H, "dh", q["w_down"]["ldT"]),
               W["dgrad_down"])
        _timed(ev, "g", lambda: gg(GMT, "dgu", "row", "w_gu", "colT", H, 2 * F, "dx", q["w_gu"]["ldT"]),
               W["dgrad_gu"])
        _timed(ev, "g", lambda: gg(GK, "dy", "colT", "hp", "colT", H, F, "dw_down", self.ldT_tok), W["wgrad_down"])
        _timed(ev, "g", lambda: gg(GK, "dgu", "colT", "xp", "colT", 2 * F, H, "dw_gu", self.ldT_tok),
               W["wgrad_gu"])


class MoeUnfusedStep:
    """The DeepSeek-V3-shaped MoE layer of MoeStep without the fused
    prologues, for comparison: the routed token rows and the down
    projection's input are given as materialised bf16 tensors, gate and up
    are separate weights and GEMMs (the nine grouped GEMMs)."""

    def __init__(self, dev, seed):
        import numpy as np

        import fp8_mixed_precision_scale_gb300 as fp8
        import synth
        self.fp8 = fp8
        E, H, F = synth.DSV3["E"], synth.DSV3["H"], synth.DSV3["F"]
        self.E, self.H, self.F = E, H, F
        sizes = synth.moe_group_sizes().numpy()
        self.sizes = sizes
        self.off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        self.off_d = torch.from_numpy(self.off).to(dev)
        self.M = M = int(self.off[-1])
        self.tokens = synth.DSV3["tokens"]
        self.name = "moe_unfused"
        self.desc = ("deepseek-v3 moe layer fwd+bwd, unfused: 4096 tokens x top-8 = 32768 routed rows (given "
                     "permuted), hidden 7168, 256 experts of ffn 2048 (gate/up/down), group sizes multinomial over "
                     "zipf(1.1) with 8 empty experts; rowwise + per-expert colwise scales; 9 grouped GEMMs")
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.tok = {"xp": _normal(g, dev, (M, H), 1.0), "hp": _normal(g, dev, (M, F), 1.0),
                    "dy_down": _normal(g, dev, (M, H), 1e-4), "dy_gate": _normal(g, dev, (M, F), 1e-4),
                    "dy_up": _normal(g, dev, (M, F), 1e-4)}
        self.tfmt = {"xp": 0, "hp": 0, "dy_down": 1, "dy_gate": 1, "dy_up": 1}
        self.w = {"w_gate": _normal(g, dev, (E * F, H), 0.02), "w_up": _normal(g, dev, (E * F, H), 0.02),
                  "w_down": _normal(g, dev, (E * H, F), 0.02)}
        self.inp = dict(self.tok, **self.w)
        self.recipe = fp8.Recipe(kind=fp8.ROWWISE)
        ldT = fp8.fp8_group_padded_offsets(self.off)[0]
        self.ldT_tok = max(16, (ldT + 15) // 16 * 16)
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            ld = r if k in self.w else self.ldT_tok
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, ld), dtype=torch.uint8, device=dev), ldT=ld,
                             srow=torch.empty(r, dtype=torch.float32, device=dev),
                             scol=torch.empty(E * c, dtype=torch.float32, device=dev))
        e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.out = {"gate": e(M, F), "up": e(M, F), "y": e(M, H), "dh": e(M, F), "dx_gate": e(M, H),
                    "dx_up": e(M, H), "dw_down": e(E, H, F), "dw_gate": e(E, F, H), "dw_up": e(E, F, H)}
        nz = int((sizes > 0).sum())
        fl = 2.0 * M * F * H
        wbytes = nz * F * H
        self.gemm_work = {  # (flops, algorithmic bytes: A + non-empty experts' weights + C)
            "fprop": (fl, M * H + wbytes + 2.0 * M * F), "fprop_down": (fl, M * F + wbytes + 2.0 * M * H),
            "dgrad_down": (fl, M * H + wbytes + 2.0 * M * F), "dgrad": (fl, M * F + wbytes + 2.0 * M * H),
            "wgrad": (fl, M * (F + H) + 2.0 * E * F * H)}
        self.flops = 9 * fl
        self.q_bytes = sum(quantize_bytes(t.shape) for t in self.inp.values())
        self.launches_per_step = 5 * len(self.tok) + 4 * len(self.w) + 9   # grouped 5, equal groups 4 launches
        self.d2h = [self.out["y"]]

    def quantize(self, k):
        t, q = self.inp[k], self.q[k]
        r, c = t.shape
        off_d = None if k in self.w else self.off_d   # expert weights: E equal groups
        f = 0 if k in self.w else self.tfmt[k]
        self.fp8.fp8_quantize(t, r, c, c, f, self.recipe, 3, None, None, q["row"], q["srow"], q["colT"],
                              q["ldT"], q["scol"], off_d, self.E)

    def run(self, ev=None, world=1):
        fp8, q, o, E, H, F, M = self.fp8, self.q, self.out, self.E, self.H, self.F, self.M
        GM, GK, GMT = fp8.GROUPED_M, fp8.GROUPED_K, fp8.GROUPED_M_BT
        off = self.off_d

        def gg(mode, a, al, fa, b, bl, fb, N, K, out, ldT=0):
            A = q[a]["row"] if al == "row" else q[a]["colT"]
            B = q[b]["row"] if bl == "row" else q[b]["colT"]
            sa = q[a]["srow"] if al == "row" else q[a]["scol"]
            sb = q[b]["srow"] if bl == "row" else q[b]["scol"]
            fp8.fp8_grouped_gemm(mode, A, fa, B, fb, off, E, M, N, K, sa, 1, sb, 1, o[out], ldT)

        W = self.gemm_work
        for k in ("xp", "w_gate", "w_up", "w_down", "hp"):
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        _timed(ev, "g", lambda: gg(GM, "xp", "row", 0, "w_gate", "row", 0, F, H, "gate"), W["fprop"])
        _timed(ev, "g", lambda: gg(GM, "xp", "row", 0, "w_up", "row", 0, F, H, "up"), W["fprop"])
        _timed(ev, "g", lambda: gg(GM, "hp", "row", 0, "w_down", "row", 0, H, F, "y"), W["fprop_down"])
        for k in ("dy_down", "dy_gate", "dy_up"):
            _timed(ev, "q", lambda k=k: self.quantize(k), quantize_bytes(self.inp[k].shape))
        _timed(ev, "g", lambda: gg(GMT, "dy_down", "row", 1, "w_down", "colT", 0, F, H, "dh",
                                   q["w_down"]["ldT"]), W["dgrad_down"])
        _timed(ev, "g", lambda: gg(GMT, "dy_gate", "row", 1, "w_gate", "colT", 0, H, F, "dx_gate",
                                   q["w_gate"]["ldT"]), W["dgrad"])
        _timed(ev, "g", lambda: gg(GMT, "dy_up", "row", 1, "w_up", "colT", 0, H, F, "dx_up",
                                   q["w_up"]["ldT"]), W["dgrad"])
        _timed(ev, "g", lambda: gg(GK, "dy_down", "colT", 1, "hp", "colT", 0, H, F, "dw_down", self.ldT_tok),
               W["wgrad"])
        _timed(ev, "g", lambda: gg(GK, "dy_gate", "colT", 1, "xp", "colT", 0, F, H, "dw_gate", self.ldT_tok),
               W["wgrad"])
        _timed(ev, "g", lambda: gg(GK, "dy_up", "colT", 1, "xp", "colT", 0, F, H, "dw_up", self.ldT_tok),
               W["wgrad"])


class MoeMxStep:
    """The DeepSeek-V3-shaped MoE layer fwd+bwd under the MXFP8 recipe, with
    the fused prologues: the token rows are gathered into expert order inside
    their quantize (fp8_mx_permute_quantize), SwiGLU of the fused gate|up
    projection's output is applied inside the quantize of the down
    projection's input (fp8_mx_swiglu_quantize); the expert weights are MX
    quantized as grouped stacks (gate and up fused per expert); six grouped
    MX GEMMs with the FLOPs of the nine unfused ones: M-grouped fprop (gate|up,
    down), M-grouped dgrad on the weights' transposed layouts, K-grouped
    wgrad."""

    def __init__(self, dev, seed):
        import numpy as np

        import fp8_mixed_precision_scale_gb300 as fp8
        import synth
        self.fp8 = fp8
        E, H, F, T = synth.DSV3["E"], synth.DSV3["H"], synth.DSV3["F"], synth.DSV3["tokens"]
        self.E, self.H, self.F = E, H, F
        sizes = synth.moe_group_sizes().numpy()
        self.off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        self.off_h = torch.from_numpy(self.off)
        self.off_d = self.off_h.to(dev)
        self.M = M = int(self.off[-1])
        self.tokens = T
        self.name = "moe_mxfp8"
        self.desc = ("deepseek-v3 moe layer fwd+bwd, mxfp8 recipe: 4096 tokens x top-8 = 32768 routed rows gathered "
                     "into expert order inside their quantize, hidden 7168, 256 experts of ffn 2048 (gate|up fused, "
                     "down), SwiGLU fused into the quantize of the down projection's input, group sizes multinomial "
                     "over zipf(1.1) with 8 empty experts; 6 grouped MX GEMMs (the FLOPs of 9)")
        rng = np.random.default_rng(seed)
        self.src = torch.from_numpy(rng.integers(0, T, size=M).astype(np.int32)).to(dev)   # routed row -> token
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.inp = {"x": _normal(g, dev, (T, H), 1.0), "w_gu": _normal(g, dev, (E * 2 * F, H), 0.02),
                    "w_down": _normal(g, dev, (E * H, F), 0.02), "dy": _normal(g, dev, (M, H), 1e-4),
                    "dgu": _normal(g, dev, (M, 2 * F), 1e-4)}
        self.P, _ = fp8.fp8_group_padded_offsets(self.off_h, fp8.MX_GROUP_ALIGN)   # padded routed rows

        def bufs(rows, cols, srows):
            return dict(row=torch.empty((rows, cols), dtype=torch.uint8, device=dev),
                        colT=torch.empty((cols, srows), dtype=torch.uint8, device=dev),
                        srow=torch.empty(fp8.fp8_mx_scale_bytes(srows, cols // 32), dtype=torch.uint8, device=dev),
                        scol=torch.empty(fp8.fp8_mx_scale_bytes(cols, srows // 32), dtype=torch.uint8, device=dev),
                        ldT=srows)
        self.q = {"xp": bufs(M, H, self.P), "hp": bufs(M, F, self.P), "dy": bufs(M, H, self.P),
                  "dgu": bufs(M, 2 * F, self.P), "w_gu": bufs(E * 2 * F, H, E * 2 * F),
                  "w_down": bufs(E * H, F, E * H)}
        e = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.out = {"gu": e(M, 2 * F), "y": e(M, H), "dh": e(M, F), "dx": e(M, H), "dw_down": e(E, H, F),
                    "dw_gu": e(E, 2 * F, H)}
        nz = int((sizes > 0).sum())
        fl = 2.0 * M * F * H
        self.gemm_work = {  # (flops, algorithmic bytes: A + non-empty experts' weights + C + scales)
            "fprop_gu": (2 * fl, M * H + 2 * nz * F * H + 4.0 * M * F + (M + 2 * nz * F) * H / 32),
            "fprop_down": (fl, M * F + nz * F * H + 2.0 * M * H + (M + nz * H) * F / 32),
            "dgrad_down": (fl, M * H + nz * F * H + 2.0 * M * F + (M + F) * H / 32),
            "dgrad_gu": (2 * fl, 2 * M * F + 2 * nz * F * H + 2.0 * M * H + (M + H) * 2 * F / 32),
            "wgrad_down": (fl, M * (F + H) + 2.0 * E * F * H + M * (F + H) / 32),
            "wgrad_gu": (2 * fl, M * (2 * F + H) + 4.0 * E * F * H + M * (2 * F + H) / 32)}
        self.flops = 9 * fl
        self.q_shapes = {"xp": (M, H), "w_gu": (E * 2 * F, H), "w_down": (E * H, F), "hp": (M, F), "dy": (M, H),
                         "dgu": (M, 2 * F)}
        self.q_bytes = sum(mx_quantize_bytes(sh) for sh in self.q_shapes.values()) + 2 * M * F
        self.launches_per_step = 6 + 6
        self.d2h = [self.out["y"]]

    def quantize(self, k):
        fp8, q = self.fp8, self.q[k]
        E = self.E
        if k == "xp":
            x = self.inp["x"]
            fp8.fp8_mx_permute_quantize(x, x.shape[0], x.shape[1], x.stride(0), self.src, self.M, 0, 3, q["row"],
                                        q["srow"], q["colT"], q["ldT"], q["scol"], self.off_d, E)
        elif k == "hp":
            gu = self.out["gu"]
            fp8.fp8_mx_swiglu_quantize(gu, self.M, self.F, gu.stride(0), 0, 3, None, 0, q["row"], q["srow"],
                                       q["colT"], q["ldT"], q["scol"], self.off_d, E)
        else:
            t = self.inp[k]
            r, c = t.shape
            # expert weights: groups of 4096 / 7168 rows, multiples of the 128-row MX group alignment, so the
            # grouped layout has no padding and equals the plain quantize of the whole stack
            off, G = (None, 0) if k.startswith("w_") else (self.off_d, E)
            f = 1 if k in ("dy", "dgu") else 0
            fp8.fp8_mx_quantize(t, r, c, c, f, 3, q["row"], q["srow"], q["colT"], q["ldT"], q["scol"], off, G)

    def run(self, ev=None, world=1):
        fp8, q, o, E, H, F, M = self.fp8, self.q, self.out, self.E, self.H, self.F, self.M
        GM, GK, GMT = fp8.GROUPED_M, fp8.GROUPED_K, fp8.GROUPED_M_BT
        off = self.off_d

        def gg(mode, a, al, fa, b, bl, fb, N, K, out, ldT=0):
            A = q[a]["row"] if al == "row" else q[a]["colT"]
            B = q[b]["row"] if bl == "row" else q[b]["colT"]
            sA = q[a]["srow"] if al == "row" else q[a]["scol"]
            sB = q[b]["srow"] if bl == "row" else q[b]["scol"]
            fp8.fp8_mx_grouped_gemm(mode, A, fa, sA, B, fb, sB, off, E, M, N, K, o[out], ldT)

        W = self.gemm_work
        for k in ("xp", "w_gu", "w_down"):
            _timed(ev, "q", lambda k=k: self.quantize(k), mx_quantize_bytes(self.q_shapes[k]))
        _timed(ev, "g", lambda: gg(GM, "xp", "row", 0, "w_gu", "row", 0, 2 * F, H, "gu"), W["fprop_gu"])
        _timed(ev, "q", lambda: self.quantize("hp"), mx_quantize_bytes(self.q_shapes["hp"]) + 2 * M * F)
        _timed(ev, "g", lambda: gg(GM, "hp", "row", 0, "w_down", "row", 0, H, F, "y"), W["fprop_down"])
        for k in ("dy", "dgu"):
            _timed(ev, "q", lambda k=k: self.quantize(k), mx_quantize_bytes(self.q_shapes[k]))
        _timed(ev, "g", lambda: gg(GMT, "dy", "row", 1, "w_down", "colT", 0, F, H, "dh", q["w_down"]["ldT"]),
               W["dgrad_down"])
        _timed(ev, "g", lambda: gg(GMT, "dgu", "row", 1, "w_gu", "colT", 0, H, 2 * F, "dx", q["w_gu"]["ldT"]),
               W["dgrad_gu"])
        _timed(ev, "g", lambda: gg(GK, "dy", "colT", 1, "hp", "colT", 0, H, F, "dw_down", self.P), W["wgrad_down"])
        _timed(ev, "g", lambda: gg(GK, "dgu", "colT", 1, "xp", "colT", 0, 2 * F, H, "dw_gu", self.P),
               W["wgrad_gu"])


# --------------------------------------------------------------------------------------------
# CPU baseline (the oracle)
# --------------------------------------------------------------------------------------------

def llama_mlp_work():
    """FLOPs and algorithmic quantize bytes of one default step."""
    flops = 0.0
    for (a, al, b, bl, o) in MLP_GEMMS:
        M, K = LLAMA_MLP_SHAPES[a][0] if al == "row" else LLAMA_MLP_SHAPES[a][0][::-1]
        N = LLAMA_MLP_SHAPES[b][0][0] if bl == "row" else LLAMA_MLP_SHAPES[b][0][1]
        flops += 2.0 * M * N * K
    q_bytes = sum(quantize_bytes(shape) for shape, _ in LLAMA_MLP_SHAPES.values())
    return {"flops": flops, "q_bytes": q_bytes}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


_CPU_INPUTS = {}


def cpu_baseline_sample(one_core=True):
    """The oracle on the default workload (the Llama-3-8B MLP block under
    delayed scaling), on the host cores:
      * the 8 quantizes of the step on their full tensors (synth's seed-1
        tensors, delayed recipe, both layouts);
      * the amax-history update of the 8 histories of length 1024;
      * the fp64 gate-projection GEMM for a block of 256 of its 8192 output
        rows, whose rate is extrapolated to the step's 9 GEMMs.
    With one_core, also on a single core (X's quantize and a 16-row GEMM
    block, extrapolated the same way)."""
    import numpy as np

    import oracle
    import synth
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    if not _CPU_INPUTS:
        base = synth.llama_mlp_base()
        _CPU_INPUTS["bits"] = {k: synth.bf16_bits(v) for k, v in base.items()}
        g = torch.Generator().manual_seed(1)
        _CPU_INPUTS["A"] = torch.randint(0, 0x70, (256, H_), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
        _CPU_INPUTS["B"] = torch.randint(0, 0x70, (F_, H_), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    bits, A, B = _CPU_INPUTS["bits"], _CPU_INPUTS["A"], _CPU_INPUTS["B"]
    w = llama_mlp_work()
    fmts = {k: (oracle.E5M2 if k.startswith("dy") else oracle.E4M3FN) for k in bits}

    def timed(threads, keys, gemm_rows):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        for k in keys:
            oracle.quantize(bits[k], fmts[k], oracle.DELAYED, scale_in=np.float32(64.0), amax_io=np.float32(0.0))
        tq = time.perf_counter() - t0
        q_bytes = sum(QUANT_BYTES_PER_ELEM * bits[k].size for k in keys)
        hist = np.zeros((8, L_HIST), np.float32)
        hist[:, 0] = 1.0
        sc, si = np.ones(8, np.float32), np.ones(8, np.float32)
        t0 = time.perf_counter()
        oracle.update_amax_history(hist, sc, si, np.array([fmts[k] for k in bits], np.uint8), oracle.MOST_RECENT, 0)
        tu = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.gemm(A[:gemm_rows], 0, B, 0, np.float32(1.0), np.float32(1.0))
        tg = time.perf_counter() - t0
        g_tflops = 2.0 * gemm_rows * F_ * H_ / tg / 1e12
        q_gbs = q_bytes / tq / 1e9
        # the oracle's step: the quantizes at their measured rate over the step's bytes, the update, the 9 GEMMs
        # at the block's rate
        step_s = w["q_bytes"] / (q_gbs * 1e9) + tu + w["flops"] / (g_tflops * 1e12)
        return {"value": w["flops"] / step_s / 1e12, "quantize_gbs": q_gbs, "update_ms": tu * 1e3,
                "gemm_gflops": g_tflops * 1e3, "step_s_extrapolated": step_s, "seconds": tq + tu + tg}

    one = timed(1, ["x"], 16) if one_core else None
    r = timed(cores, list(bits), 256)
    out = {"value": r["value"], "unit": "TFLOP/s", "cores": cores, "cpu": cpu_model(), "kind": "oracle",
           "sample": (f"oracle on the step's 8 quantizes, full tensors ({r['quantize_gbs']:.3f} GB/s, timed), the "
                      f"8 x 1024 history update ({r['update_ms']:.2f} ms, timed) and the fp64 gate GEMM for 256 of "
                      f"its 8192 output rows [256x14336x4096] ({r['gemm_gflops']:.2f} GFLOP/s, timed), the GEMM "
                      f"rate extrapolated to the step's 9 GEMMs: {r['step_s_extrapolated']:.1f} s per step"),
           "quantize_gbs": r["quantize_gbs"], "update_ms": r["update_ms"], "gemm_gflops": r["gemm_gflops"],
           "step_s_extrapolated": r["step_s_extrapolated"], "seconds": r["seconds"] + (one["seconds"] if one else 0)}
    if one:
        out["one_core"] = {"value": one["value"], "quantize_gbs": one["quantize_gbs"], "gemm_gflops": one["gemm_gflops"],
                           "sample": "X's quantize [8192x4096] and a 16-row gate GEMM block, extrapolated likewise"}
    return out


# --------------------------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------------------------

def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def _max_over_ranks(v, world, dev):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def _category(ev, kind):
    items = ev.get(kind, [])
    return [a.elapsed_time(b) for a, b, _ in items], [w for _, _, w in items]


def run_gpu(args, rank, world, local_rank):
    import fp8_mixed_precision_scale_gb300 as fp8
    from fp8_mixed_precision_scale_gb300 import build as fp8build
    if rank == 0 or world == 1:
        fp8build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    fp8.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hbm_gbs = peaks()[0]

    if args.workload in ("gemm", "quantize", "grouped_m", "grouped_k", "mx_grouped_m", "mx_grouped_k",
                         "quantize_grouped", "mx_gemm", "mx_quantize", "mx_permute", "mx_swiglu", "permute", "swiglu",
                         "bw_quantize", "rowwise_quantize", "rowwise_resident", "stack_quantize", "mx_stack_quantize"):
        run_single_kernel(args, dev, rank)
        return
    if args.workload == "sweep":
        run_sweep(args, dev, rank, hbm_gbs)
        return
    step = make_step(args.workload, dev, 1 + rank)
    m = measure(step, args.steps, args.warmup, world, local_rank, dev, graph=args.workload in GRAPH_STEPS)
    e2e = run_e2e(step, args, world, dev)
    out = {
        "metric": METRIC,
        "value": m["value"],
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": m["ms_per_step"],
        "ms_per_step_eager": m["ms_per_step_eager"],
        "ms_per_step_graph": m["ms_per_step_graph"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8 e4m3/e5m2 operands, fp32 accumulate, bf16 out",
        "data": "synthetic",
        "config": {"workload": step.desc, "name": step.name, "tokens_per_rank": step.tokens,
                   "parallelism": f"dp{world}",
                   "l2": "inputs larger than L2 (GBs of operands touched per step), no flush needed",
                   "timing": "CUDA events on the launching stream, max over ranks; the step launched eagerly "
                             "and replayed from a CUDA graph, the faster reported"},
        "tokens_per_s": m["tokens_per_s"],
        "gemm": m["gemm"],
        "quantize": m["quantize"],
        "update_us": m["update_us"],
        "roofline": m["roofline"],
        "e2e": e2e,
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": m["clocks"],
    }
    del step
    torch.cuda.empty_cache()
    if args.workload == "llama_mlp" and world == 1 and not args.no_configs:
        out["configs"] = run_configs(args, dev, local_rank, m)
    if args.workload == "llama_mlp" and rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_sample()
    if rank == 0:
        print(json.dumps(out), flush=True)


STEPS = {"llama_mlp": lambda dev, seed: llama_mlp_step(dev, seed), "flux": lambda dev, seed: flux_step(dev, seed),
         "llama_rowwise": lambda dev, seed: RowwiseStep(dev, seed), "moe": lambda dev, seed: MoeStep(dev, seed),
         "moe_unfused": lambda dev, seed: MoeUnfusedStep(dev, seed), "llama_mxfp8": lambda dev, seed: MxStep(dev, seed),
         "llama_blockwise": lambda dev, seed: MxStep(dev, seed, recipe="blockwise"),
         "moe_mxfp8": lambda dev, seed: MoeMxStep(dev, seed), "tiny": lambda dev, seed: TinyStep(dev, seed)}


def make_step(name, dev, seed):
    return STEPS[name](dev, seed)


# steps also timed replayed from a CUDA graph (the faster of the two step
# times is reported, both are printed): the dense-layer steps, whose launches
# are a visible share of the step; the MoE steps run long kernels
GRAPH_STEPS = ("tiny", "llama_mlp", "llama_rowwise", "flux", "llama_mxfp8", "llama_blockwise")


def measure(step, steps, warmup, world, local_rank, dev, graph=False):
    """Warm up, then time `steps` steps with CUDA events on the launching
    stream (barrier + synchronize on both sides, max over ranks), with the
    clocks sampled inside the timed window; per-category kernel times from
    events around every launch.  The FP8 tensor peak is 2 x the measured
    bf16 peak: the burst figure, or the sustained one when the power cap
    acted during the window (sw_power_cap among the throttle reasons).  With
    graph, the step is also captured once in a CUDA graph and replayed, and
    the faster of the two step times is reported (the per-category kernel
    times stay those of the eager launches)."""
    import fp8_mixed_precision_scale_gb300 as fp8
    hbm_gbs, bf16_burst, bf16_sust, peak_src = peaks()
    for _ in range(max(3, warmup)):
        step.run(world=world)
    assert fp8.fp8_sync_status() == 0

    sampler = ClockSampler(local_rank)
    ev = {}
    _barrier(world)
    sampler.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t_start.record()
    for _ in range(steps):
        step.run(ev, world=world)
    t_end.record()
    _barrier(world)
    st = fp8.fp8_sync_status()
    assert st == 0, f"device status {st}"
    ms_step = _max_over_ranks(t_start.elapsed_time(t_end), world, dev) / steps
    ms_eager = ms_step
    graph_ms = None
    if graph and world == 1:
        # the same step replayed from a CUDA graph (inside the clock window):
        # removes the host's launch cost and the gaps between launches
        s_cap = torch.cuda.Stream()
        s_cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_cap):
            step.run()
        torch.cuda.current_stream().wait_stream(s_cap)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, capture_error_mode="relaxed"):
            step.run()
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        t_start.record()
        for _ in range(steps):
            cg.replay()
        t_end.record()
        torch.cuda.synchronize()
        assert fp8.fp8_sync_status() == 0
        graph_ms = t_start.elapsed_time(t_end) / steps
        ms_step = min(ms_step, graph_ms)
    w1 = time.time()
    clocks = sampler.stop((w0, w1))

    capped = bool(clocks and "sw_power_cap" in clocks.get("reasons", []))
    fp8_burst, fp8_sust = 2.0 * bf16_burst, 2.0 * bf16_sust
    fp8_peak = fp8_sust if capped else fp8_burst
    peak_name = "sustained" if capped else "burst"
    g_ms, g_work = _category(ev, "g")
    q_ms, q_work = _category(ev, "q")
    u_ms, _ = _category(ev, "u")
    gemm_tflops = sum(f for f, _ in g_work) / (sum(g_ms) * 1e-3) / 1e12
    # roofline time of every GEMM launch: max(flops / tensor peak, bytes / HBM)
    g_roof_ms = sum(max(f / (fp8_peak * 1e12), b / (hbm_gbs * 1e9)) * 1e3 for f, b in g_work)
    g_tensor_ms = sum(f / (fp8_peak * 1e12) * 1e3 for f, _ in g_work)
    g_frac = g_roof_ms / sum(g_ms)
    q_gbs = sum(q_work) / (sum(q_ms) * 1e-3) / 1e9 if q_ms else 0.0

    # the dominant kernel category of the step gives the roofline object
    if sum(g_ms) >= sum(q_ms):
        if g_roof_ms <= g_tensor_ms * 1.0001:      # tensor-bound GEMMs
            roof = {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                    "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                    "frac_burst": round(gemm_tflops / fp8_burst, 4), "frac_sustained": round(gemm_tflops / fp8_sust, 4),
                    "kernel": "mx_gemm_kernel" if isinstance(step, (MxStep, MoeMxStep)) else "fp8_gemm_pair_kernel",
                    "traffic": gemm_traffic(step.name),
                    "peak_source": f"{peak_src}: 2 x {peak_name} bf16 {bf16_sust if capped else bf16_burst} TFLOP/s "
                                   f"(fp8/bf16 nominal ratio 2; {peak_name} because sw_power_cap was "
                                   f"{'' if capped else 'not '}seen in the timed window)"}
        else:                                      # HBM-bound (grouped GEMMs at the MoE shape)
            gbs = sum(b for _, b in g_work) / (sum(g_ms) * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                    "frac": round(g_frac, 4), "traffic": None,
                    "kernel": "mx_gemm_kernel (grouped)" if isinstance(step, MoeMxStep) else "fp8_gemm_kernel (grouped)",
                    "peak_source": f"{peak_src} HBM copy bandwidth; frac = roofline time max(flops / fp8 {peak_name} "
                                   f"peak, bytes / HBM) over the measured time"}
    else:
        roof = {"bound": "hbm", "achieved": round(q_gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(q_gbs / hbm_gbs, 4), "traffic": None, "kernel": "quantize (amax + cast)",
                "peak_source": f"{peak_src} HBM copy bandwidth"}
    return {
        "ms_per_step": round(ms_step, 4),
        "ms_per_step_eager": round(ms_eager, 4),
        "ms_per_step_graph": round(graph_ms, 4) if graph_ms is not None else None,
        "value": round(world * step.flops / (ms_step * 1e-3) / 1e12, 2),
        "tokens_per_s": round(world * step.tokens / (ms_step * 1e-3), 1),
        "gemm": {"ms_per_step": round(sum(g_ms) / steps, 4), "tflops": round(gemm_tflops, 1),
                 "frac_of_fp8_peak": round(gemm_tflops / fp8_peak, 4),
                 "frac_of_fp8_burst": round(gemm_tflops / fp8_burst, 4),
                 "frac_of_fp8_sustained": round(gemm_tflops / fp8_sust, 4),
                 "frac_of_roofline": round(g_frac, 4), "launches_per_step": len(g_ms) // steps},
        "quantize": {"ms_per_step": round(sum(q_ms) / steps, 4), "gbs": round(q_gbs, 1),
                     "frac_of_hbm": round(q_gbs / hbm_gbs, 4), "bytes_per_step": step.q_bytes,
                     "calls_per_step": len(q_ms) // steps},
        "update_us": round(1e3 * sum(u_ms) / len(u_ms), 2) if u_ms else None,
        "roofline": roof,
        "clocks": clocks,
    }


def run_configs(args, dev, local_rank, headline):
    """Every configuration of the benchmark set, each measured like the
    headline step on this GPU: the tiny rowwise linear, the Llama-3-8B MLP
    block under delayed scaling (the headline itself), the Llama-3-8B
    attention projections + MLP under the rowwise recipe, the DeepSeek-V3 MoE
    layer, the Flux-12B linears, and the knee of the 2^20 .. 2^30-element
    quantize sweep."""
    hbm_gbs = peaks()[0]
    out = {}
    summary = lambda name, step, m: {  # noqa: E731
        "workload": step.desc, "ms_per_step": m["ms_per_step"], "tflops": m["value"],
        "tokens_per_s": m["tokens_per_s"], "gemm_tflops": m["gemm"]["tflops"],
        "gemm_frac_of_roofline": m["gemm"]["frac_of_roofline"], "quantize_gbs": m["quantize"]["gbs"],
        "quantize_frac_of_hbm": m["quantize"]["frac_of_hbm"], "update_us": m["update_us"],
        "roofline": {k: m["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac")},
        "clocks": m["clocks"]}
    for cfg, name, steps in (("1_tiny", "tiny", 200), ("3_llama_rowwise", "llama_rowwise", 20),
                             ("4_dsv3_moe", "moe", 10), ("5_flux", "flux", 20)):
        step = make_step(name, dev, 1)
        m = measure(step, steps, 3, 1, local_rank, dev, graph=name in GRAPH_STEPS)
        out[cfg] = summary(name, step, m)
        if name == "tiny":
            out[cfg]["us_per_step"] = round(m["ms_per_step"] * 1e3, 2)
            out[cfg]["l2"] = "inputs inside L2: launch-bound, reported in us; the step replayed from a CUDA graph"
        del step
        torch.cuda.empty_cache()
    out["2_llama_mlp_delayed"] = {"workload": LLAMA_MLP_DESC, "note": "the headline line itself",
                                  "ms_per_step": headline["ms_per_step"], "tflops": headline["value"],
                                  "tokens_per_s": headline["tokens_per_s"],
                                  "gemm_tflops": headline["gemm"]["tflops"],
                                  "quantize_gbs": headline["quantize"]["gbs"],
                                  "quantize_frac_of_hbm": headline["quantize"]["frac_of_hbm"],
                                  "roofline": {k: headline["roofline"][k]
                                               for k in ("bound", "achieved", "peak", "unit", "frac")}}
    pts = sweep_points(dev, hbm_gbs, max_reps=40)
    knee = next((pt["elements"] for pt in pts if pt["frac_of_hbm"] >= 0.8), None)
    best = max(pts, key=lambda pt: pt["gbs"])
    out["5_quantize_sweep"] = {"workload": "delayed quantize, e4m3fn, both layouts, x ~ N(0,1) [n/4096, 4096], "
                                           "n = 2^20 .. 2^30",
                               "knee_elements": knee, "best_gbs": best["gbs"], "best_frac_of_hbm": best["frac_of_hbm"],
                               "points": [{k: pt[k] for k in ("elements", "us_per_launch", "gbs", "frac_of_hbm")}
                                          for pt in pts]}
    return out


def run_e2e(step, args, world, dev):
    """The same metric through the public API with host buffers: every step
    copies that step's bf16 inputs from pinned host memory to the device and
    reads the forward output back, inside the timed region.  The copies run
    on a second stream into a second set of input buffers, so the transfer of
    step i + 1 overlaps the kernels of step i (as a training input pipeline
    would)."""
    # pinned buffers on the NUMA node the GPU is attached to: allocated and
    # first touched by this thread while it runs on that node's cores
    numa = gpu_numa(dev)
    saved = os.sched_getaffinity(0)
    if numa.get("cpus"):
        os.sched_setaffinity(0, numa["cpus"])
    try:
        pinned = {k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for k, t in step.inp.items()}
        for k in pinned:
            pinned[k].copy_(step.inp[k])
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in step.d2h]
    finally:
        os.sched_setaffinity(0, saved)
    # the host link on its own: the step's H2D copies back to back
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record()
    for k in pinned:
        step.inp[k].copy_(pinned[k], non_blocking=True)
    h1.record()
    torch.cuda.synchronize()
    h2d_gbs = sum(t.numel() * t.element_size() for t in pinned.values()) / (h0.elapsed_time(h1) * 1e-3) / 1e9
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    n = 2 if step.name.startswith("moe") else max(3, min(args.steps, 10))
    sets = [dict(step.inp), {k: torch.empty_like(t) for k, t in step.inp.items()}]
    comp = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]   # inputs of a set copied
    free = [torch.cuda.Event(), torch.cuda.Event()]    # compute done with a set
    done = torch.cuda.Event()
    for e in free:
        e.record(comp)

    def copy_in(i):
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(free[i % 2])
            for k in pinned:
                sets[i % 2][k].copy_(pinned[k], non_blocking=True)
            ready[i % 2].record(copy_s)

    def compute(i):
        comp.wait_event(ready[i % 2])
        step.inp = sets[i % 2]
        step.run(world=world)
        free[i % 2].record(comp)
        for h, d in zip(host_out, step.d2h):
            h.copy_(d, non_blocking=True)

    copy_in(0)
    compute(0)
    _barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    copy_s.wait_event(e0)
    copy_in(1)
    for i in range(1, n + 1):
        if i + 1 <= n:
            copy_in(i + 1)
        compute(i)
    done.record(comp)
    e1.record(comp)
    _barrier(world)
    step.inp = sets[0]
    ms = _max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
    return {"value": round(world * step.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "overlap": "H2D of step i+1 on a second stream during the kernels of step i",
            "h2d_gbs": round(h2d_gbs, 1), "host_link_bound_ms": round(h2d / (h2d_gbs * 1e9) * 1e3, 3),
            "pinned_numa": {k: v for k, v in numa.items() if k != "cpus"}}


def gpu_numa(dev):
    """The NUMA node of the GPU's PCI function and that node's cores (those
    this process may run on), from sysfs; empty when unknown."""
    try:
        p = torch.cuda.get_device_properties(dev)
        dom, bus, slot = getattr(p, "pci_domain_id"), getattr(p, "pci_bus_id"), getattr(p, "pci_device_id")
        addr = f"{dom:04x}:{bus:02x}:{slot:02x}.0"
        with open(f"/sys/bus/pci/devices/{addr}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return {"pci": addr, "node": None}
        cpus = set()
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return {"pci": addr, "node": node, "cpus": cpus, "cores_on_node": len(cpus)}
    except Exception as e:   # noqa: BLE001  (no sysfs entry, older torch): report and go on
        return {"node": None, "error": type(e).__name__}


def sweep_points(dev, hbm_gbs, max_reps=200):
    """Delayed quantize (E4M3, both layouts) of 2^20 .. 2^30 elements: GB/s
    against size, inputs rotated over buffers larger than L2."""
    import fp8_mixed_precision_scale_gb300 as fp8
    import synth
    rec = fp8.Recipe(kind=fp8.DELAYED)
    scale = torch.full((1,), 64.0, device=dev)
    amax = torch.zeros(1, device=dev)
    points = []
    for p in range(20, 31):
        n = 1 << p
        rows, cols = n // 4096, 4096
        # rotate over enough buffers that one round touches more than 3 x L2
        nbuf = max(1, -(-(400 << 20) // (4 * n)))
        base = synth.sweep_tensor(n, dev)
        bufs = []
        for i in range(nbuf):
            bufs.append((base if i == 0 else base.clone(), torch.empty((rows, cols), dtype=torch.uint8, device=dev),
                         torch.empty((cols, rows), dtype=torch.uint8, device=dev),
                         torch.empty(1, device=dev), torch.empty(1, device=dev)))
        reps = max(nbuf, min(max_reps, (64 << 30) // (4 * n)))

        def launch(i):
            x, qr, qc, sr, sc = bufs[i % nbuf]
            fp8.fp8_quantize(x, rows, cols, cols, 0, rec, 3, scale, amax, qr, sr, qc, rows, sc)
        for i in range(nbuf + 3):
            launch(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(reps):
            launch(i)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        gbs = 4.0 * n / (ms * 1e-3) / 1e9
        points.append({"elements": n, "us_per_launch": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                       "frac_of_hbm": round(gbs / hbm_gbs, 4), "buffers": nbuf, "launches": reps})
        del bufs, base
        torch.cuda.empty_cache()
    assert fp8.fp8_sync_status() == 0
    return points


def run_sweep(args, dev, rank, hbm_gbs):
    """Delayed quantize (E4M3, both layouts) of 2^20 .. 2^30 elements."""
    import fp8_mixed_precision_scale_gb300 as fp8
    points = sweep_points(dev, hbm_gbs)
    assert fp8.fp8_sync_status() == 0
    knee = next((pt["elements"] for pt in points if pt["frac_of_hbm"] >= 0.8), None)
    best = max(points, key=lambda pt: pt["gbs"])
    if rank == 0:
        print(json.dumps({"metric": METRIC, "workload": "sweep", "value": best["gbs"], "unit": "GB/s",
                          "config": {"workload": "delayed quantize e4m3fn, both layouts, x ~ N(0,1) shaped "
                                                 "[n/4096, 4096], n = 2^20..2^30; buffers rotated so each round "
                                                 "exceeds L2", "algorithmic_bytes_per_element": 4},
                          "knee_elements_at_80pct": knee, "points": points}), flush=True)


def grouped_case(kind, dev, E=64, rows=8192):
    """A reduced DeepSeek-V3 expert GEMM for profiling: 64 experts (2 empty),
    8192 routed rows, hidden 7168, ffn 2048; random FP8 operands."""
    import numpy as np

    import fp8_mixed_precision_scale_gb300 as fp8
    import synth
    H, F = synth.DSV3["H"], synth.DSV3["F"]
    sizes = synth.moe_group_sizes(total_rows=rows, E=E, n_forced_empty=2).numpy()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    off_d = torch.from_numpy(off).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)

    def codes(*shape):
        return (torch.randn(shape, generator=g, device=dev) * 64).clamp(-448, 448).to(
            torch.float8_e4m3fn).view(torch.uint8)
    s_rows, s_ef, s_eh = (torch.ones(n, device=dev) for n in (rows, E * F, E * H))
    if kind == "grouped_m":       # fprop of the gate projection
        A, B, C = codes(rows, H), codes(E, F, H), torch.empty((rows, F), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8.fp8_grouped_gemm(fp8.GROUPED_M, A, 0, B, 0, off_d, E, rows, F, H, s_rows, 1,  # noqa
                                          s_ef, 1, C, 0)
        wbytes = int((sizes > 0).sum()) * F * H
        return fn, (rows * H + wbytes + 2.0 * rows * F) / 1e9, "GB/s (algorithmic)"
    if kind == "mx_grouped_m":    # MXFP8 fprop of the gate projection (MX-quantized routed rows and weights)
        gb = torch.Generator(device=dev)
        gb.manual_seed(9)
        x = torch.randn((rows, H), generator=gb, device=dev).to(torch.bfloat16)
        w = (torch.randn((E * F, H), generator=gb, device=dev) * 0.02).to(torch.bfloat16)
        qa = fp8.mx_quantize(x, 0, fp8.LAYOUT_ROW, group_offsets=off_d, host_offsets=torch.from_numpy(off))
        qw = fp8.mx_quantize(w, 0, fp8.LAYOUT_ROW)
        C = torch.empty((rows, F), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8.fp8_mx_grouped_gemm(fp8.GROUPED_M, qa.q_row, 0, qa.s_row, qw.q_row, 0, qw.s_row,  # noqa
                                             off_d, E, rows, F, H, C, 0)
        wbytes = int((sizes > 0).sum()) * F * H
        return fn, (rows * H + wbytes + 2.0 * rows * F) / 1e9, "GB/s (algorithmic)"
    if kind == "mx_grouped_k":    # MXFP8 wgrad of the gate projection from grouped MX quantizes
        gb = torch.Generator(device=dev)
        gb.manual_seed(8)
        dy = torch.randn((rows, F), generator=gb, device=dev).to(torch.bfloat16)
        x = torch.randn((rows, H), generator=gb, device=dev).to(torch.bfloat16)
        off_h = torch.from_numpy(off)
        qa = fp8.mx_quantize(dy, 0, fp8.LAYOUT_COLT, group_offsets=off_d, host_offsets=off_h)
        qb = fp8.mx_quantize(x, 0, fp8.LAYOUT_COLT, group_offsets=off_d, host_offsets=off_h)
        C = torch.empty((E, F, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8.fp8_mx_grouped_gemm(fp8.GROUPED_K, qa.q_colT, 0, qa.s_col, qb.q_colT, 0, qb.s_col,  # noqa
                                             off_d, E, rows, F, H, C, qa.ld_colT)
        return fn, (rows * (F + H) + 2.0 * E * F * H) / 1e9, "GB/s (algorithmic)"
    ldT = int(fp8.fp8_group_padded_offsets(off)[0])
    ldT = (ldT + 15) // 16 * 16
    A, B = codes(F, ldT), codes(H, ldT)   # wgrad of the gate projection: dW_e = dY_e^T X_e
    C = torch.empty((E, F, H), dtype=torch.bfloat16, device=dev)
    fn = lambda: fp8.fp8_grouped_gemm(fp8.GROUPED_K, A, 1, B, 0, off_d, E, rows, F, H, s_ef, 1,  # noqa
                                      s_eh, 1, C, ldT)
    return fn, (rows * (F + H) + 2.0 * E * F * H) / 1e9, "GB/s (algorithmic)"


def grouped_weight_quantize_case(dev, E=64):
    """Rowwise quantize of one reduced MoE gate weight [64 * 2048, 7168] with
    per-expert column scales (64 equal groups), for profiling."""
    import fp8_mixed_precision_scale_gb300 as fp8
    import synth
    H, F = synth.DSV3["H"], synth.DSV3["F"]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    w = _normal(g, dev, (E * F, H), 0.02)
    rows = E * F
    q_row = torch.empty((rows, H), dtype=torch.uint8, device=dev)
    q_colT = torch.empty((H, rows), dtype=torch.uint8, device=dev)
    sr = torch.empty(rows, device=dev)
    sc = torch.empty(E * H, device=dev)
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    # equal groups (no offsets): the form the MoE steps quantize their expert weights in
    fn = lambda: fp8.fp8_quantize(w, rows, H, H, 0, rec, 3, None, None, q_row, sr, q_colT, rows, sc,  # noqa: E731
                                  None, E)
    return fn, quantize_bytes((rows, H)) / 1e9, "GB/s (algorithmic)"


def weight_stack_case(kind, stack, dev):
    """Quantize of a whole DeepSeek-V3 expert-weight stack (256 experts,
    gate|up fused: [256 x 4096, 7168]; down: [256 x 7168, 2048]), both
    layouts, as the MoE steps quantize their weights: rowwise with 256 equal
    groups (`stack_quantize`) or MX (`mx_stack_quantize`)."""
    import fp8_mixed_precision_scale_gb300 as fp8
    import synth
    E, H, F = synth.DSV3["E"], synth.DSV3["H"], synth.DSV3["F"]
    rows, cols = (E * 2 * F, H) if stack == "gateup" else (E * H, F)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    w = _normal(g, dev, (rows, cols), 0.02)
    if kind == "mx_stack_quantize":
        q = fp8.mx_quantize(w, 0)
        fn = lambda: fp8.fp8_mx_quantize(w, rows, cols, cols, 0, 3, q.q_row, q.s_row, q.q_colT,  # noqa: E731
                                         q.ld_colT, q.s_col)
        return fn, rows * cols * (2 + 2 + 2 / 32) / 1e9, "GB/s (algorithmic)"
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    q_colT = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    sr = torch.empty(rows, device=dev)
    sc = torch.empty(E * cols, device=dev)
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    fn = lambda: fp8.fp8_quantize(w, rows, cols, cols, 0, rec, 3, None, None, q_row, sr, q_colT, rows, sc,  # noqa: E731
                                  None, E)
    return fn, quantize_bytes((rows, cols)) / 1e9, "GB/s (algorithmic)"


def moe_fused_case(kind, dev, T=4096, topk=8, E=256):
    """DeepSeek-V3-shaped fused MoE prologue + MX quantize (both layouts,
    per-expert grouping): `mx_permute` gathers 4096 tokens x top-8 routed
    rows of hidden 7168 into expert order; `mx_swiglu` applies SwiGLU to the
    [32768, 2 x 2048] gate|up output.  Returns (fused fn, unfused-chain fn,
    algorithmic GB per call)."""
    import numpy as np

    import fp8_mixed_precision_scale_gb300 as fp8
    import synth
    H, F = synth.DSV3["H"], synth.DSV3["F"]
    rng = np.random.default_rng(5)
    experts = np.argsort(rng.random((T, E)), axis=1)[:, :topk]
    tok = np.repeat(np.arange(T), topk)
    order = np.argsort(experts.reshape(-1), kind="stable")
    src = torch.from_numpy(tok[order].astype(np.int32)).to(dev)
    off_h = torch.from_numpy(np.concatenate([[0], np.cumsum(np.bincount(experts.reshape(-1), minlength=E))])
                             .astype(np.int32))
    off = off_h.to(dev)
    rows = T * topk
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    if kind == "mx_permute":
        x = _normal(g, dev, (T, H), 1.0)
        fused = lambda: fp8.mx_permute_quantize(x, src, 0, 3, group_offsets=off, host_offsets=off_h)  # noqa: E731
        src64 = src.long()
        unfused = lambda: fp8.mx_quantize(x.index_select(0, src64), 0, 3, group_offsets=off,  # noqa: E731
                                          host_offsets=off_h)
        return fused, unfused, rows * H * (2 + 2 + 2 / 32) / 1e9
    if kind == "permute":   # rowwise recipe, per-expert column scales
        x = _normal(g, dev, (T, H), 1.0)
        fused = lambda: fp8.permute_quantize(x, src, 0, off, off_h)  # noqa: E731
        src64 = src.long()
        rec = fp8.Recipe(kind=fp8.ROWWISE)
        unfused = lambda: fp8.quantize(x.index_select(0, src64), 0, rec, group_offsets=off,  # noqa: E731
                                       host_offsets=off_h)
        return fused, unfused, rows * H * 4 / 1e9
    gu = _normal(g, dev, (rows, 2 * F), 2.0)
    if kind == "swiglu":    # rowwise recipe, per-expert column scales
        fused = lambda: fp8.swiglu_quantize(gu, 0, off, off_h)  # noqa: E731
        rec = fp8.Recipe(kind=fp8.ROWWISE)

        def unfused_rw():
            h = (torch.nn.functional.silu(gu[:, :F].float()) * gu[:, F:].float()).to(torch.bfloat16)
            return fp8.quantize(h, 0, rec, group_offsets=off, host_offsets=off_h)
        return fused, unfused_rw, rows * F * (4 + 2) / 1e9
    fused = lambda: fp8.mx_swiglu_quantize(gu, 0, 3, group_offsets=off, host_offsets=off_h)  # noqa: E731

    def unfused():
        h = (torch.nn.functional.silu(gu[:, :F].float()) * gu[:, F:].float()).to(torch.bfloat16)
        return fp8.mx_quantize(h, 0, 3, group_offsets=off, host_offsets=off_h)
    return fused, unfused, rows * F * (4 + 2 + 2 / 32) / 1e9


def run_single_kernel(args, dev, rank):
    """Time one kernel of the default step in isolation (profiling aid)."""
    import fp8_mixed_precision_scale_gb300 as fp8
    unfused = None
    if args.workload in ("mx_permute", "mx_swiglu", "permute", "swiglu"):
        fn, unfused, work = moe_fused_case(args.workload, dev)
        unit = "GB/s (algorithmic)"
    elif args.workload in ("grouped_m", "grouped_k", "mx_grouped_m", "mx_grouped_k"):
        fn, work, unit = grouped_case(args.workload, dev)
    elif args.workload == "quantize_grouped":
        fn, work, unit = grouped_weight_quantize_case(dev)
    elif args.workload in ("stack_quantize", "mx_stack_quantize"):
        fn, work, unit = weight_stack_case(args.workload, args.stack, dev)
    elif args.workload == "mx_gemm":
        step = MxStep(dev, 1, keys=("x", "w_gate"), outs=("gate",))
        for k in ("x", "w_gate"):
            step.quantize(k)
        fn = lambda: step.gemm(*MLP_GEMMS[0])  # noqa: E731
        work, unit = step.gemm_work["gate"][0] / 1e12, "TFLOP/s"
    elif args.workload == "rowwise_quantize":
        step = RowwiseStep(dev, 1, keys=("dy_gate",))
        fn = lambda: step.quantize("dy_gate")  # noqa: E731
        work, unit = quantize_bytes(step.inp["dy_gate"].shape) / 1e9, "GB/s (algorithmic)"
    elif args.workload == "rowwise_resident":
        # X [8192, 4096] is 64 MB: the calls rotate over three copies (192 MB,
        # more than L2) so no call starts with its input in L2
        step = RowwiseStep(dev, 1, keys=("x",))
        copies = [step.inp["x"]] + [step.inp["x"].clone() for _ in range(2)]
        turn = [0]

        def rotate(f):
            step.inp["x"] = copies[turn[0] % 3]
            turn[0] += 1
            f("x")
        fn = lambda: rotate(step.quantize_resident)  # noqa: E731
        work, unit = quantize_bytes(step.inp["x"].shape) / 1e9, "GB/s (algorithmic)"
        unfused = lambda: rotate(step.quantize)  # noqa: E731
    elif args.workload in ("mx_quantize", "bw_quantize"):
        step = MxStep(dev, 1, keys=("dy_gate",), outs=(), recipe="mxfp8" if args.workload == "mx_quantize" else "blockwise")
        fn = lambda: step.quantize("dy_gate")  # noqa: E731
        work, unit = mx_quantize_bytes(step.inp["dy_gate"].shape) / 1e9, "GB/s"
    elif args.workload == "gemm":
        step = llama_mlp_step(dev, 1, keys=("x", "w_gate"), outs=("gate",))
        for k in ("x", "w_gate"):   # real FP8 operands for the GEMM
            step.quantize(k)
        fn = lambda: step.gemm(*MLP_GEMMS[0])  # noqa: E731
        work, unit = step.gemm_work["gate"][0] / 1e12, "TFLOP/s"
    else:
        step = llama_mlp_step(dev, 1, keys=("dy_gate",), outs=())
        fn = lambda: step.quantize("dy_gate")  # noqa: E731
        work, unit = quantize_bytes(step.inp["dy_gate"].shape) / 1e9, "GB/s"
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    ms = a.elapsed_time(b) / args.steps
    line = {"workload": args.workload, "ms_per_launch": round(ms, 4), "value": round(work / (ms * 1e-3), 1),
            "unit": unit, "launches": args.steps}
    if unfused is not None:   # the same result through the unfused chain of separate launches
        for _ in range(3):
            unfused()
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            unfused()
        b.record()
        torch.cuda.synchronize()
        line["unfused_chain_ms"] = round(a.elapsed_time(b) / args.steps, 4)
        line["speedup_vs_chain"] = round(line["unfused_chain_ms"] / ms, 2)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only): each
    step is the bounded sample of cpu_baseline_sample (the step's quantizes
    and update in full, one 256-row block of a GEMM); ms_per_step is that
    sample's wall time, value the oracle's rate extrapolated to the whole
    step."""
    if rank != 0:
        return
    t0 = time.perf_counter()
    vals, secs = [], []
    base = None
    for i in range(max(0, args.warmup) + args.steps):
        s0 = time.perf_counter()
        b = cpu_baseline_sample(one_core=False)   # the host-core rate only: keeps the run to a few minutes
        if i >= args.warmup:
            vals.append(b["value"])
            secs.append(time.perf_counter() - s0)
        base = b
    value = statistics.mean(vals)
    wall = time.perf_counter() - t0
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(secs), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": LLAMA_MLP_DESC, "parallelism": "host cores",
                   "step": "the bounded sample described in cpu_baseline.sample"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": base["cores"], "cpu": base["cpu"],
                         "kind": "oracle", "sample": base["sample"]},
        "oracle_step_s_extrapolated": round(base["step_s_extrapolated"], 1),
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration measurements")
    ap.add_argument("--stack", default="gateup", choices=["gateup", "down"],
                    help="stack_quantize / mx_stack_quantize: which DeepSeek-V3 expert-weight stack")
    ap.add_argument("--workload", default="llama_mlp",
                    choices=["llama_mlp", "llama_rowwise", "llama_mxfp8", "llama_blockwise", "moe", "moe_unfused",
                             "moe_mxfp8", "flux", "tiny",
                             "sweep",
                             "gemm", "quantize", "bw_quantize", "rowwise_quantize", "rowwise_resident",
                             "grouped_m", "grouped_k", "mx_grouped_m", "mx_grouped_k", "quantize_grouped", "mx_gemm",
                             "mx_quantize",
                             "mx_permute",
                             "mx_swiglu", "permute", "swiglu", "stack_quantize", "mx_stack_quantize"],
                    help="llama_mlp: the whole fwd+bwd FP8 step of the Llama-3-8B MLP (default); see the "
                         "module docstring for the others")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if args.steps < 1:
            args.steps = 1
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
