"""Seeded synthetic inputs for the FP8 linear-layer workloads.

This module only draws random numbers: it holds none of the method's
arithmetic (no amax, no scale, no cast).  Both the CPU oracle's tests and the
CUDA library's tests and benchmark take their inputs from here, so the two
sides always see the same bf16 tensors.

Recipe (all tensors bf16, drawn in fp32 then rounded to bf16 by torch):
  * tiny          seed 0  X [256,512] ~ N(0,1) with 0.1% of entries (131,
                          chosen by a seeded permutation) multiplied by 50;
                          W [512,512] ~ N(0,0.02); dY [256,512] ~ N(0,1e-3).
  * llama_mlp     seed 1  tokens 8192, hidden 4096, ffn 14336.  Acts ~ N(0,1),
                          weights ~ N(0,0.02), grads ~ N(0,1e-4).  The SwiGLU
                          output H [8192,14336] is drawn directly.
  * llama_attn    seed 2  as llama_mlp plus QKV [6144,4096] and O [4096,6144]
                          weights; activations Student-t with nu = 4.  The
                          MLP of this (rowwise) workload: seed 102, the
                          llama_mlp shapes with Student-t (nu = 4)
                          activations X and H.
  * dsv3_moe      seed 3  4096 tokens x top-8 = 32768 routed rows, hidden
                          7168, 256 experts of ffn 2048.  Group sizes
                          ~ Multinomial(32768, p), p_e ~ r_e^-1.1 over a seeded
                          permutation r of 1..256, with 8 seeded experts given
                          p = 0 (empty groups).
  * flux          seed 4  tokens 2 x (4096 + 512) = 9216, hidden 3072, MLP
                          3072 -> 12288 -> 3072, QKV 3072 -> 9216.
Drift over steps (delayed-scaling runs): step t multiplies activations by
2^(t/25), gradients by 2^(-t/25) and weights by 1 + 0.002 t; at t = 30 the
activations are multiplied by a further 8 (one-step spike).  The drifted
tensor is bf16(fp32(base) * g_t).
"""
from __future__ import annotations

import math

import torch

TINY = dict(T=256, H=512, seed=0)
LLAMA = dict(T=8192, H=4096, F=14336, QKV=6144, seed_mlp=1, seed_attn=2)
DSV3 = dict(tokens=4096, topk=8, H=7168, E=256, F=2048, seed=3, n_forced_empty=8, zipf_s=1.1)
FLUX = dict(T=9216, H=3072, F=12288, QKV=9216, seed=4)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std, g, device="cpu") -> torch.Tensor:
    """N(0, std) in fp32, rounded to bf16."""
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def student_t(shape, nu: int, g, device="cpu") -> torch.Tensor:
    """Student-t with integer nu: z / sqrt(chi2_nu / nu), chi2 from nu squared normals."""
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi += torch.randn(shape, generator=g, device=device, dtype=torch.float32).square()
    return (z / torch.sqrt(chi / nu)).to(torch.bfloat16)


def tiny(device="cpu"):
    """Tiny FP8 linear (rowwise recipe): X with outliers, W, dY."""
    g = _gen(TINY["seed"])
    T, H = TINY["T"], TINY["H"]
    x = torch.randn((T, H), generator=g, dtype=torch.float32)
    n_out = round(0.001 * T * H)
    idx = torch.randperm(T * H, generator=g)[:n_out]
    x.view(-1)[idx] *= 50.0
    w = torch.randn((H, H), generator=g, dtype=torch.float32) * 0.02
    dy = torch.randn((T, H), generator=g, dtype=torch.float32) * 1e-3
    out = dict(x=x.to(torch.bfloat16), w=w.to(torch.bfloat16), dy=dy.to(torch.bfloat16))
    return {k: v.to(device) for k, v in out.items()}


def llama_mlp_base(device="cpu", scale_down: int = 1):
    """Base tensors of the Llama-3-8B MLP block (before drift).

    scale_down > 1 divides T, H and F by it (same distributions) for fast
    parity runs that keep the structure.
    """
    g = _gen(LLAMA["seed_mlp"])
    T, H, F = LLAMA["T"] // scale_down, LLAMA["H"] // scale_down, LLAMA["F"] // scale_down
    t = dict(
        x=normal((T, H), 1.0, g),
        w_gate=normal((F, H), 0.02, g),
        w_up=normal((F, H), 0.02, g),
        w_down=normal((H, F), 0.02, g),
        h=normal((T, F), 1.0, g),          # SwiGLU output (down-proj input), drawn directly
        dy_down=normal((T, H), 1e-4, g),   # grad of the block output
        dy_gate=normal((T, F), 1e-4, g),   # grad of the gate-proj output
        dy_up=normal((T, F), 1e-4, g),     # grad of the up-proj output
    )
    return {k: v.to(device) for k, v in t.items()}


ACT_KEYS = ("x", "h")
GRAD_KEYS = ("dy_down", "dy_gate", "dy_up")
WEIGHT_KEYS = ("w_gate", "w_up", "w_down", "w_qkv", "w_o")


def drift_factor(key: str, t: int) -> float:
    """Multiplier of base tensor `key` at step t (see the module docstring)."""
    if key in ACT_KEYS or key.startswith("x"):
        g = 2.0 ** (t / 25.0)
        if t == 30:
            g *= 8.0
        return g
    if key.startswith("dy"):
        return 2.0 ** (-t / 25.0)
    return 1.0 + 0.002 * t


def drifted(base: torch.Tensor, key: str, t: int) -> torch.Tensor:
    """bf16(fp32(base) * g_t)."""
    return (base.float() * drift_factor(key, t)).to(torch.bfloat16)


def llama_attn_extra(device="cpu", scale_down: int = 1):
    """Attention-projection tensors of the rowwise Llama-3-8B workload."""
    g = _gen(LLAMA["seed_attn"])
    T, H, Q = LLAMA["T"] // scale_down, LLAMA["H"] // scale_down, LLAMA["QKV"] // scale_down
    t = dict(
        x=student_t((T, H), 4, g),
        w_qkv=normal((Q, H), 0.02, g),
        o_in=student_t((T, Q), 4, g),      # attention output = O-proj input
        w_o=normal((H, Q), 0.02, g),
        dy_qkv=normal((T, Q), 1e-4, g),
        dy_o=normal((T, H), 1e-4, g),
    )
    return {k: v.to(device) for k, v in t.items()}


def llama_rowwise_mlp(device="cpu", scale_down: int = 1):
    """MLP tensors of the rowwise Llama-3-8B workload: the llama_mlp shapes,
    Student-t (nu = 4) activations, N(0, 0.02) weights, N(0, 1e-4) grads."""
    g = _gen(LLAMA["seed_attn"] + 100)
    T, H, F = LLAMA["T"] // scale_down, LLAMA["H"] // scale_down, LLAMA["F"] // scale_down
    t = dict(
        x=student_t((T, H), 4, g),
        w_gate=normal((F, H), 0.02, g),
        w_up=normal((F, H), 0.02, g),
        w_down=normal((H, F), 0.02, g),
        h=student_t((T, F), 4, g),
        dy_down=normal((T, H), 1e-4, g),
        dy_gate=normal((T, F), 1e-4, g),
        dy_up=normal((T, F), 1e-4, g),
    )
    return {k: v.to(device) for k, v in t.items()}


def moe_group_sizes(total_rows=None, E=None, seed=None, n_forced_empty=None, s=None):
    """Expert group sizes of the DeepSeek-V3-shaped MoE layer (int64 [E])."""
    total_rows = total_rows or DSV3["tokens"] * DSV3["topk"]
    E = E or DSV3["E"]
    seed = DSV3["seed"] if seed is None else seed
    n_forced_empty = DSV3["n_forced_empty"] if n_forced_empty is None else n_forced_empty
    s = DSV3["zipf_s"] if s is None else s
    g = _gen(seed)
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    p = rank.pow(-s)
    empty = torch.randperm(E, generator=g)[:n_forced_empty]
    p[empty] = 0.0
    p = p / p.sum()
    draws = torch.multinomial(p, total_rows, replacement=True, generator=g)
    return torch.bincount(draws, minlength=E).to(torch.int64)


def offsets_from_sizes(sizes) -> torch.Tensor:
    off = torch.zeros(len(sizes) + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.as_tensor(sizes, dtype=torch.int64), 0).to(torch.int32)
    return off


def moe_tokens(device="cpu", rows=None, H=None, F=None, seed=None):
    """Token-side tensors of the MoE layer: permuted acts, down input, grads."""
    g = _gen((DSV3["seed"] if seed is None else seed) + 1000)
    rows = rows or DSV3["tokens"] * DSV3["topk"]
    H, F = H or DSV3["H"], F or DSV3["F"]
    t = dict(
        xp=normal((rows, H), 1.0, g),
        hp=normal((rows, F), 1.0, g),
        dy_down=normal((rows, H), 1e-4, g),
        dy_gate=normal((rows, F), 1e-4, g),
        dy_up=normal((rows, F), 1e-4, g),
    )
    return {k: v.to(device) for k, v in t.items()}


def moe_weight(shape, device="cpu", seed=None) -> torch.Tensor:
    """Expert weights ~ N(0, 0.02).  Large ones are drawn on the target device."""
    s = (DSV3["seed"] if seed is None else seed) + 2000
    dev = torch.device(device)
    g = _gen(s, device=dev)
    return normal(shape, 0.02, g, device=dev)


def flux_base(device="cpu", scale_down: int = 1):
    g = _gen(FLUX["seed"])
    T, H, F, Q = (FLUX[k] // scale_down for k in ("T", "H", "F", "QKV"))
    t = dict(
        x=normal((T, H), 1.0, g),
        w_qkv=normal((Q, H), 0.02, g),
        w_up=normal((F, H), 0.02, g),
        h=normal((T, F), 1.0, g),
        w_down=normal((H, F), 0.02, g),
        dy_qkv=normal((T, Q), 1e-4, g),
        dy_up=normal((T, F), 1e-4, g),
        dy_down=normal((T, H), 1e-4, g),
    )
    return {k: v.to(device) for k, v in t.items()}


def sweep_tensor(n_elems: int, device="cpu", seed: int = 4) -> torch.Tensor:
    """Quantize-sweep input: n elements ~ N(0,1) shaped [n / 4096, 4096]."""
    assert n_elems % 4096 == 0
    dev = torch.device(device)
    g = _gen(seed, device=dev)
    return normal((n_elems // 4096, 4096), 1.0, g, device=dev)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a (CPU) bf16 tensor."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def randomize_special(t: torch.Tensor, g: torch.Generator, frac: float = 0.01) -> torch.Tensor:
    """Sprinkle zeros, -0, huge values, tiny values and bf16 subnormals into t."""
    flat = t.clone().view(-1)
    n = flat.numel()
    k = max(1, int(n * frac))
    vals = torch.tensor([0.0, -0.0, 3.0e38, -3.0e38, 1e-40, -1e-40, 1e-30, 65504.0, 1e5, -1e5],
                        dtype=torch.float32).to(torch.bfloat16)
    idx = torch.randperm(n, generator=g)[:k]
    pick = torch.randint(0, vals.numel(), (k,), generator=g)
    flat[idx] = vals[pick].to(flat.device)
    return flat.view_as(t)


def isqrt_ceil(x: int) -> int:
    return int(math.ceil(math.sqrt(x)))
