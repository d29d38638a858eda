"""Benchmark of the FP8 linear hot path on one GB300 (or N, one process each).

One step = the whole FP8 path of the Llama-3-8B MLP block (tokens 8192,
hidden 4096, ffn 14336) under delayed scaling with the hybrid format:
  8 fused quantizes (X, W_gate, W_up, W_down, H, dY_down, dY_gate, dY_up;
    E4M3 forward / E5M2 gradients; rowwise + colwise-transposed layouts),
  9 FP8 GEMMs (fprop, dgrad, wgrad of gate, up and down; 962 GFLOP each),
  1 fused amax-history update (8 histories of length 1024, most_recent).
Under torchrun each rank runs its own batch (data parallel, weak scaling);
the one exchange of the path -- a MAX all-reduce of the 8 current amaxes
before the update -- goes over NCCL.

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
T_, H_, F_ = 8192, 4096, 14336
L_HIST = 1024
GEMM_FLOP = 2.0 * T_ * H_ * F_            # every GEMM of the block has the same M*N*K
N_GEMM = 9
QUANT_ELEMS = {"x": T_ * H_, "w_gate": F_ * H_, "w_up": F_ * H_, "w_down": H_ * F_, "h": T_ * F_,
               "dy_down": T_ * H_, "dy_gate": T_ * F_, "dy_up": T_ * F_}
QUANT_BYTES_PER_ELEM = 4                  # 2 B read + 1 B per layout, two layouts
WORKLOAD = ("llama3-8b-mlp fwd+bwd, delayed scaling: tokens 8192, hidden 4096, ffn 14336, "
            "hybrid e4m3 fwd / e5m2 grads, amax history 1024 most_recent, margin 0")

# DRAM bytes (read + write) of one dense GEMM launch, the gate projection
# 8192x14336x4096, from one ncu capture (profiles/fp8_gemm_kernel_llama_gate_8192x14336x4096.md).
# Reported only while the profiled sources are unchanged.
GEMM_TRAFFIC = {"bytes": 291.5e6,
                "sources": {"gemm.cu": "bdce445243241ecb", "fp8gb_device.cuh": "ea559f4d3db429bb"}}


def gemm_traffic():
    import hashlib
    csrc = os.path.join(ROOT, "fp8_mixed_precision_scale_gb300", "csrc")
    for name, want in GEMM_TRAFFIC["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != want:
                return None
    return GEMM_TRAFFIC["bytes"]


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
# the GPU arm
# --------------------------------------------------------------------------------------------

class MlpStep:
    """Buffers and the launch sequence of one FP8 fwd+bwd step of the MLP block."""

    SHAPES = {"x": ((T_, H_), 1.0), "w_gate": ((F_, H_), 0.02), "w_up": ((F_, H_), 0.02),
              "w_down": ((H_, F_), 0.02), "h": ((T_, F_), 1.0), "dy_down": ((T_, H_), 1e-4),
              "dy_gate": ((T_, F_), 1e-4), "dy_up": ((T_, F_), 1e-4)}
    OUTS = {"gate": (T_, F_), "up": (T_, F_), "y": (T_, H_), "dh": (T_, F_), "dx_gate": (T_, H_),
            "dx_up": (T_, H_), "dw_down": (H_, F_), "dw_gate": (F_, H_), "dw_up": (F_, H_)}

    def __init__(self, dev, seed: int, keys=None, outs=None):
        """keys / outs restrict the tensors allocated (single-kernel workloads)."""
        import fp8_mixed_precision_scale_gb300 as fp8
        self.fp8 = fp8
        g = torch.Generator(device=dev)
        g.manual_seed(seed)

        def normal(shape, std):
            return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

        self.order = list(self.SHAPES.keys())
        self.inp = {k: normal(*self.SHAPES[k]) for k in self.order if keys is None or k in keys}
        self.fmt = {k: (fp8.E5M2 if k.startswith("dy") else fp8.E4M3FN) for k in self.order}
        n = len(self.order)
        self.hist = torch.zeros((n, L_HIST), dtype=torch.float32, device=dev)
        self.scale = torch.ones(n, dtype=torch.float32, device=dev)
        self.scale_inv = torch.ones(n, dtype=torch.float32, device=dev)
        self.fmt_dev = torch.tensor([self.fmt[k] for k in self.order], dtype=torch.uint8, device=dev)
        self.q = {}
        for k, t in self.inp.items():
            r, c = t.shape
            self.q[k] = dict(row=torch.empty((r, c), dtype=torch.uint8, device=dev),
                             colT=torch.empty((c, r), dtype=torch.uint8, device=dev),
                             srow=torch.empty(1, dtype=torch.float32, device=dev),
                             scol=torch.empty(1, dtype=torch.float32, device=dev))
        self.out = {k: torch.empty(shape, dtype=torch.bfloat16, device=dev) for k, shape in self.OUTS.items()
                    if outs is None or k in outs}
        self.recipe = fp8.Recipe(kind=fp8.DELAYED, margin=0, history_len=L_HIST, algo=fp8.MOST_RECENT)
        # launches per step: 8 quantize (1 kernel each, delayed) + 9 GEMMs + 1 update
        self.launches_per_step = 8 + 9 + 1

    def quantize(self, k, i):
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

    GEMMS = [  # (A, A layout, B, B layout, output)
        ("x", "row", "w_gate", "row", "gate"),          # fprop gate
        ("x", "row", "w_up", "row", "up"),              # fprop up
        ("h", "row", "w_down", "row", "y"),             # fprop down
        ("dy_down", "row", "w_down", "colT", "dh"),     # dgrad down
        ("dy_gate", "row", "w_gate", "colT", "dx_gate"),  # dgrad gate
        ("dy_up", "row", "w_up", "colT", "dx_up"),      # dgrad up
        ("dy_down", "colT", "h", "colT", "dw_down"),    # wgrad down
        ("dy_gate", "colT", "x", "colT", "dw_gate"),    # wgrad gate
        ("dy_up", "colT", "x", "colT", "dw_up"),        # wgrad up
    ]

    def run(self, ev=None, world=1):
        """One step.  ev: optional dict of event lists to time the quantize and GEMM launches."""
        idx = {k: i for i, k in enumerate(self.order)}
        fwd_q = ["x", "w_gate", "w_up", "w_down", "h"]
        bwd_q = ["dy_down", "dy_gate", "dy_up"]
        for k in fwd_q:
            self._timed(ev, "q", lambda k=k: self.quantize(k, idx[k]))
        for g in self.GEMMS[:3]:
            self._timed(ev, "g", lambda g=g: self.gemm(*g))
        for k in bwd_q:
            self._timed(ev, "q", lambda k=k: self.quantize(k, idx[k]))
        for g in self.GEMMS[3:]:
            self._timed(ev, "g", lambda g=g: self.gemm(*g))
        if world > 1:
            from fp8_mixed_precision_scale_gb300 import dp
            dp.reduce_current_amax(self.hist)
        self._timed(ev, "u", lambda: self.fp8.fp8_update_amax_history(
            self.hist, self.scale, self.scale_inv, self.fmt_dev, len(self.order), L_HIST, self.fp8.MOST_RECENT, 0))

    @staticmethod
    def _timed(ev, kind, fn):
        if ev is None:
            fn()
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ev[kind].append((a, b))


def cpu_baseline_sample():
    """The oracle on a bounded sample of the same workload, on the host cores."""
    import numpy as np

    import oracle
    import synth
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    g = torch.Generator().manual_seed(1)
    x = (torch.randn((2048, H_), generator=g)).to(torch.bfloat16)            # 2048 of the 8192 token rows of X
    xb = synth.bf16_bits(x)
    t0 = time.perf_counter()
    oracle.quantize(xb, oracle.E4M3FN, oracle.DELAYED, scale_in=np.float32(64.0), amax_io=np.float32(0.0))
    tq = time.perf_counter() - t0
    q_gbs = QUANT_BYTES_PER_ELEM * x.numel() / tq / 1e9
    # GEMM: 8 full output rows of the gate projection (K = 4096, N = 14336)
    A = torch.randint(0, 0x70, (8, H_), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    B = torch.randint(0, 0x70, (F_, H_), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    t0 = time.perf_counter()
    oracle.gemm(A, 0, B, 0, np.float32(1.0), np.float32(1.0))
    tg = time.perf_counter() - t0
    flops = 2.0 * 8 * F_ * H_
    g_tflops = flops / tg / 1e12
    # the step-time model of the oracle: 9 GEMMs at its GEMM rate + 8 quantizes at its quantize rate
    step_s = N_GEMM * GEMM_FLOP / (g_tflops * 1e12) + sum(QUANT_ELEMS.values()) * QUANT_BYTES_PER_ELEM / (q_gbs * 1e9)
    value = N_GEMM * GEMM_FLOP / step_s / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": (f"oracle delayed quantize (both layouts) of X rows 0..2047 [2048x4096] "
                       f"({q_gbs:.3f} GB/s) and the fp64 gate GEMM for 8 output rows [8x14336x4096] "
                       f"({g_tflops * 1e3:.4f} GFLOP/s), extrapolated to one whole step"),
            "quantize_gbs": q_gbs, "gemm_tflops": g_tflops, "seconds": tq + tg}


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
    hbm_gbs, bf16_burst, bf16_sust, peak_src = peaks()
    fp8_peak = 2.0 * bf16_sust               # FP8 dense = 2x bf16 dense (nominal 4.5 vs 2.25 PFLOP/s)

    if args.workload == "gemm":
        run_single_kernel(args, MlpStep(dev, seed=1 + rank, keys=("x", "w_gate"), outs=("gate",)), rank, world)
        return
    if args.workload == "quantize":
        run_single_kernel(args, MlpStep(dev, seed=1 + rank, keys=("dy_gate",), outs=()), rank, world)
        return
    step = MlpStep(dev, seed=1 + rank)
    for _ in range(max(3, args.warmup)):
        step.run(world=world)
    assert fp8.fp8_sync_status() == 0

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    ev = {"q": [], "g": [], "u": []}
    barrier()
    sampler.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t_start.record()
    for _ in range(args.steps):
        step.run(ev, world=world)
    t_end.record()
    barrier()
    w1 = time.time()
    clocks = sampler.stop((w0, w1))
    st = fp8.fp8_sync_status()
    assert st == 0, f"device status {st}"
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt)
    ms_step = total_ms / args.steps
    g_ms = [a.elapsed_time(b) for a, b in ev["g"]]
    q_ms = [a.elapsed_time(b) for a, b in ev["q"]]
    u_ms = [a.elapsed_time(b) for a, b in ev["u"]]
    gemm_avg_ms = sum(g_ms) / len(g_ms)
    gemm_tflops = GEMM_FLOP / (gemm_avg_ms * 1e-3) / 1e12
    q_bytes = sum(QUANT_ELEMS.values()) * QUANT_BYTES_PER_ELEM
    q_ms_step = sum(q_ms) / args.steps
    q_gbs = q_bytes / (q_ms_step * 1e-3) / 1e9

    # end to end through the public API with host buffers: H2D of the step's
    # inputs from pinned memory, the step, D2H of the block output and dX
    pinned = {k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for k, t in step.inp.items()}
    for k in pinned:
        pinned[k].copy_(step.inp[k])
    host_y = torch.empty(step.out["y"].shape, dtype=torch.bfloat16, pin_memory=True)
    host_dx = torch.empty(step.out["dx_gate"].shape, dtype=torch.bfloat16, pin_memory=True)
    host_scale = torch.empty(len(step.order), dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = host_y.numel() * 2 + host_dx.numel() * 2 + host_scale.numel() * 4
    e2e_steps = max(2, min(args.steps, 5))

    def e2e_step():
        for k in pinned:
            step.inp[k].copy_(pinned[k], non_blocking=True)
        step.run(world=world)
        host_y.copy_(step.out["y"], non_blocking=True)
        host_dx.copy_(step.out["dx_gate"], non_blocking=True)
        host_scale.copy_(step.scale, non_blocking=True)
    e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    e1.record()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt)

    value = world * N_GEMM * GEMM_FLOP / (ms_step * 1e-3) / 1e12
    e2e_value = world * N_GEMM * GEMM_FLOP / (e2e_ms * 1e-3) / 1e12
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8 e4m3/e5m2 operands, fp32 accumulate, bf16 out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_rank": T_, "parallelism": f"dp{world}",
                   "l2": "inputs larger than L2 (about 2.4 GB of operands touched per step)",
                   "timing": "CUDA events on the launching stream, max over ranks"},
        "tokens_per_s": round(world * T_ / (ms_step * 1e-3), 1),
        "gemm": {"avg_ms": round(gemm_avg_ms, 4), "tflops": round(gemm_tflops, 1),
                 "frac_of_fp8_peak": round(gemm_tflops / fp8_peak, 4)},
        "quantize": {"ms_per_step": round(q_ms_step, 4), "gbs": round(q_gbs, 1),
                     "frac_of_hbm": round(q_gbs / hbm_gbs, 4), "bytes_per_elem": QUANT_BYTES_PER_ELEM},
        "update_us": round(1e3 * sum(u_ms) / len(u_ms), 2),
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4), "traffic": gemm_traffic(),
                     "peak_source": f"{peak_src}: 2 x sustained bf16 {bf16_sust} TFLOP/s (fp8/bf16 nominal ratio 2)"},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_sample()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_single_kernel(args, step, rank, world):
    """Time one kernel of the step in isolation (profiling aid)."""
    import fp8_mixed_precision_scale_gb300 as fp8
    if args.workload == "gemm":
        for k in ("x", "w_gate"):   # real FP8 operands for the GEMM
            step.quantize(k, step.order.index(k))
        fn = lambda: step.gemm(*MlpStep.GEMMS[0])  # noqa: E731
        work, unit = GEMM_FLOP / 1e12, "TFLOP/s"
    else:
        fn = lambda: step.quantize("dy_gate", step.order.index("dy_gate"))  # noqa: E731
        work, unit = QUANT_ELEMS["dy_gate"] * QUANT_BYTES_PER_ELEM / 1e9, "GB/s"
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
    if rank == 0:
        print(json.dumps({"workload": args.workload, "ms_per_launch": round(ms, 4),
                          "value": round(work / (ms * 1e-3), 1), "unit": unit, "launches": args.steps}), flush=True)


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    t0 = time.perf_counter()
    vals = []
    base = None
    for i in range(max(0, args.warmup) + args.steps):
        b = cpu_baseline_sample()
        if i >= args.warmup:
            vals.append(b["value"])
        base = b
    value = statistics.mean(vals)
    wall = time.perf_counter() - t0
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * N_GEMM * GEMM_FLOP / (value * 1e12),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": base["cores"], "kind": "oracle",
                         "sample": base["sample"]},
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
    ap.add_argument("--workload", default="llama_mlp", choices=["llama_mlp", "gemm", "quantize"],
                    help="llama_mlp: the whole fwd+bwd FP8 step (default); gemm / quantize: one kernel of it "
                         "(the gate-projection GEMM 8192x14336x4096, the delayed quantize of a [8192, 14336] "
                         "tensor), for profiling")
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
