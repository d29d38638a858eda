"""CPU oracle for the FP8 linear-layer hot path (test infrastructure only).

This package wraps ``fp8_oracle.c`` -- a plain, slow, scalar C restatement of
what the path computes -- through ctypes and numpy.  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the CUDA library and
its Python binding never do, and this package imports nothing from them.

Sources of each definition are cited in ``fp8_oracle.c``:
  * "FP8 training for Flux models" (Configuration > Key FP8 Parameters): the
    recipe knobs -- format, recipe, margin, amax history length, amax compute
    algorithm.
  * "FP8 Training on MI300X" ("Discovered AMD FP8 dtype difference", "Patched
    nanochat/fp8.py"): E4M3 forward / E5M2 backward, e4m3fn max 448 against
    e4m3fnuz max 240; float8_e5m2fnuz as AMD's backward format.
  * "How PyTorch FP8 Optimizations on AMD GPUs ..." (What Happened) and "FP8
    Training on AMD GPUs with TorchTitan and TorchAO": rowwise scaling,
    colwise scales with a transposed layout, grouped GEMM for MoE.
  * MXFP8 (the "mxfp8" recipe of the Flux page; MXFP8 grouped GEMM on the
    TorchTitan/TorchAO page): the OCP Microscaling v1.0 definition -- blocks
    of 32, E8M0 scale 2^(floor(log2 amax) - emax_elem).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3FN, E5M2, E4M3FNUZ, E5M2FNUZ = 0, 1, 2, 3
DELAYED, TENSORWISE, ROWWISE = 0, 1, 2
MOST_RECENT, MAX = 0, 1
LAYOUT_ROW, LAYOUT_COLT = 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C11, no FMA contraction, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
            lib.orc_set_threads.restype = None
            lib.orc_set_threads.argtypes = [i32]
            lib.orc_fp8_decode.restype = f64
            lib.orc_fp8_decode.argtypes = [i32, i32]
            lib.orc_fp8_encode.restype = i32
            lib.orc_fp8_encode.argtypes = [f64, i32]
            lib.orc_fp8_max_code.restype = i32
            lib.orc_fp8_max_code.argtypes = [i32]
            lib.orc_fp8_nan_code.restype = i32
            lib.orc_fp8_nan_code.argtypes = [i32]
            lib.orc_fp8_max_value.restype = f64
            lib.orc_fp8_max_value.argtypes = [i32]
            lib.orc_current_scale.restype = None
            lib.orc_current_scale.argtypes = [f32, i32, i32, P, P]
            lib.orc_padded_offsets.restype = i64
            lib.orc_padded_offsets.argtypes = [P, i32, P]
            lib.orc_quantize.restype = i32
            lib.orc_quantize.argtypes = [P, i64, i64, i64, i32, i32, i32, i32, P, P, P, P, P, P, P, i32]
            lib.orc_amax_bf16.restype = f32
            lib.orc_amax_bf16.argtypes = [P, i64, i64, i64]
            lib.orc_cast_points.restype = None
            lib.orc_cast_points.argtypes = [P, P, i64, i32, P]
            lib.orc_update_amax_history.restype = None
            lib.orc_update_amax_history.argtypes = [P, P, P, P, i32, i32, i32, i32, P]
            lib.orc_gemm.restype = None
            lib.orc_gemm.argtypes = [P, i32, i64, P, i32, i64, i64, i64, i64, P, i32, P, i32,
                                     P, P, i64, P, P]
            lib.orc_grouped_gemm.restype = None
            lib.orc_grouped_gemm.argtypes = [i32, P, i32, P, i32, P, i32, i64, i64, i64, P, i32,
                                             P, i32, P, P, P, i64, P, P]
            lib.orc_mx_emax.restype = i32
            lib.orc_mx_emax.argtypes = [i32]
            lib.orc_mx_scale_code.restype = i32
            lib.orc_mx_scale_code.argtypes = [f64, i32]
            lib.orc_e8m0_decode.restype = f64
            lib.orc_e8m0_decode.argtypes = [i32]
            lib.orc_padded_offsets_align.restype = i64
            lib.orc_padded_offsets_align.argtypes = [P, i32, i64, P]
            lib.orc_mx_quantize.restype = i32
            lib.orc_mx_quantize.argtypes = [P, i64, i64, i64, i32, i32, P, i32, i64, P, P, P, i64, P]
            lib.orc_mx_gemm.restype = None
            lib.orc_mx_gemm.argtypes = [P, i32, i64, P, i64, P, i32, i64, P, i64, i64, i64, i64, P, P, i64,
                                        P, P]
            lib.orc_bf16_from_double.restype = ctypes.c_uint16
            lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
            lib.orc_swiglu_bf16.restype = None
            lib.orc_swiglu_bf16.argtypes = [P, P, i64, P]
            lib.orc_blockwise_code.restype = i32
            lib.orc_blockwise_code.argtypes = [f64, i32]
            lib.orc_blockwise_quantize.restype = i32
            lib.orc_blockwise_quantize.argtypes = [P, i64, i64, i64, i32, i32, i32, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- codec ---------------------------------------------------------------

def fp8_decode(code: int, fmt: int) -> float:
    return _load().orc_fp8_decode(int(code), int(fmt))


def fp8_encode(v: float, fmt: int) -> int:
    """Round an fp32 value (given as a Python float) to the nearest code."""
    return _load().orc_fp8_encode(float(np.float32(v)), int(fmt))


def fp8_max_code(fmt: int) -> int:
    return _load().orc_fp8_max_code(int(fmt))


def fp8_nan_code(fmt: int) -> int:
    return _load().orc_fp8_nan_code(int(fmt))


def fp8_max_value(fmt: int) -> float:
    return _load().orc_fp8_max_value(int(fmt))


def decode_table(fmt: int) -> np.ndarray:
    return np.array([fp8_decode(c, fmt) for c in range(256)], dtype=np.float64)


def current_scale(amax: float, fmt: int, margin: int = 0):
    s, si = ctypes.c_float(), ctypes.c_float()
    _load().orc_current_scale(float(np.float32(amax)), fmt, margin, ctypes.byref(s), ctypes.byref(si))
    return np.float32(s.value), np.float32(si.value)


# --- quantize ------------------------------------------------------------

def padded_offsets(offsets) -> np.ndarray:
    off = _c(offsets, np.int32)
    G = off.size - 1
    poff = np.zeros(G + 1, dtype=np.int64)
    _load().orc_padded_offsets(_ptr(off), G, _ptr(poff))
    return poff


def quantize(x_bits, fmt, kind, margin=0, layouts=LAYOUT_ROW | LAYOUT_COLT, scale_in=None,
             amax_io=None, offsets=None):
    """Quantize a bf16 matrix given as its uint16 bit patterns [rows, cols].

    Returns a dict with q_row [rows, cols] u8, scale_inv_row, q_colT
    [cols, ldT] u8, scale_inv_col, amax (the value left in amax_io).
    """
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    G = 0 if offsets is None else len(offsets) - 1
    off = None if offsets is None else _c(offsets, np.int32)
    ldT = rows if off is None else int(padded_offsets(off)[-1])
    q_row = np.zeros((rows, cols), np.uint8) if layouts & LAYOUT_ROW else None
    q_colT = np.zeros((cols, ldT), np.uint8) if layouts & LAYOUT_COLT else None
    if kind == ROWWISE:
        sr = np.zeros(rows, np.float32)
        sc = np.zeros((G, cols) if off is not None else cols, np.float32)
    else:
        sr = np.zeros(1, np.float32)
        sc = np.zeros(1, np.float32)
    sin = None if scale_in is None else _c(np.atleast_1d(scale_in), np.float32)
    amax = np.array([0.0 if amax_io is None else amax_io], np.float32)
    _load().orc_quantize(_ptr(x), rows, cols, cols, fmt, kind, margin, layouts, _ptr(sin), _ptr(amax),
                         _ptr(q_row), _ptr(sr), _ptr(q_colT), _ptr(sc), _ptr(off), G)
    return dict(q_row=q_row, scale_inv_row=sr, q_colT=q_colT, scale_inv_col=sc, amax=np.float32(amax[0]))


def amax_bf16(x_bits) -> np.float32:
    x = _c(x_bits, np.uint16)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    return np.float32(_load().orc_amax_bf16(_ptr(x), x.shape[0], x.shape[1], x.shape[1]))


def cast_points(x_bits, scales, fmt) -> np.ndarray:
    """encode(fp32(x[i]) * scales[i]) for selected elements."""
    x = _c(x_bits, np.uint16).ravel()
    s = _c(np.broadcast_to(np.asarray(scales, np.float32), x.shape), np.float32)
    out = np.zeros(x.size, np.uint8)
    _load().orc_cast_points(_ptr(x), _ptr(s), x.size, fmt, _ptr(out))
    return out


# --- history update ------------------------------------------------------

def update_amax_history(hist, scale, scale_inv, fmt, algo, margin, nonfinite=None):
    """In-place update of numpy arrays hist [n, L], scale [n], scale_inv [n]."""
    assert hist.dtype == np.float32 and hist.flags.c_contiguous
    n, L = hist.shape
    fm = _c(np.broadcast_to(np.asarray(fmt, np.uint8), (n,)), np.uint8)
    _load().orc_update_amax_history(_ptr(hist), _ptr(scale), _ptr(scale_inv), _ptr(fm), n, L, algo, margin,
                                    _ptr(nonfinite))


# --- GEMM ------------------------------------------------------------------

def gemm(A, fa, B, fb, sa, sb, points=None):
    """Dequantised TN GEMM in double.  A [M, K] u8, B [N, K] u8.

    sa / sb: scalar (one scale) or vector [M] / [N].  points: optional
    (pm, pn) int arrays.  Returns (ref, bound) as float64 arrays ([M, N] or
    [npts]).
    """
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    sa_a = _c(np.atleast_1d(sa), np.float32)
    sb_a = _c(np.atleast_1d(sb), np.float32)
    if points is None:
        ref = np.zeros((M, N)); bound = np.zeros((M, N)); pm = pn = None; npts = 0
    else:
        pm = _c(points[0], np.int64); pn = _c(points[1], np.int64); npts = pm.size
        ref = np.zeros(npts); bound = np.zeros(npts)
    _load().orc_gemm(_ptr(A), fa, K, _ptr(B), fb, K, M, N, K, _ptr(sa_a), int(sa_a.size > 1),
                     _ptr(sb_a), int(sb_a.size > 1), _ptr(pm), _ptr(pn), npts, _ptr(ref), _ptr(bound))
    return ref, bound


def grouped_gemm(mode, A, fa, B, fb, offsets, N, K, sa, sb, pg, pm, pn):
    """Sampled grouped GEMM (see orc_grouped_gemm).  Returns (ref, bound)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    off = _c(offsets, np.int32)
    G = off.size - 1
    sa_a = _c(np.atleast_1d(sa), np.float32)
    sb_a = _c(np.atleast_1d(sb), np.float32)
    pm = _c(pm, np.int64); pn = _c(pn, np.int64)
    pg = _c(pg if pg is not None else np.zeros_like(pm), np.int64)
    ref = np.zeros(pm.size); bound = np.zeros(pm.size)
    _load().orc_grouped_gemm(mode, _ptr(A), fa, _ptr(B), fb, _ptr(off), G, int(off[-1]), N, K,
                             _ptr(sa_a), int(sa_a.size > 1), _ptr(sb_a), int(sb_a.size > 1),
                             _ptr(pg), _ptr(pm), _ptr(pn), pm.size, _ptr(ref), _ptr(bound))
    return ref, bound


# --- MXFP8 -------------------------------------------------------------------

MX_BLOCK = 32


def mx_emax(fmt: int) -> int:
    return _load().orc_mx_emax(int(fmt))


def mx_scale_code(amax: float, fmt: int) -> int:
    """E8M0 code of a block whose largest magnitude is amax."""
    return _load().orc_mx_scale_code(float(amax), int(fmt))


def e8m0_decode(code: int) -> float:
    return _load().orc_e8m0_decode(int(code))


def padded_offsets_align(offsets, align: int) -> np.ndarray:
    off = _c(offsets, np.int32)
    G = off.size - 1
    poff = np.zeros(G + 1, dtype=np.int64)
    _load().orc_padded_offsets_align(_ptr(off), G, int(align), _ptr(poff))
    return poff


def mx_quantize(x_bits, fmt, layouts=LAYOUT_ROW | LAYOUT_COLT, offsets=None, align=128):
    """MX quantize of a bf16 matrix given as uint16 bits [rows, cols].

    Returns dict(q_row [rows, cols], s_row [SR, cols/32], q_colT [cols, P],
    s_col [cols, P/32]) with plain row-major E8M0 scale matrices; SR = P =
    rows (ungrouped) or the total of the group sizes padded to `align`.
    """
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    G = 0 if offsets is None else len(offsets) - 1
    off = None if offsets is None else _c(offsets, np.int32)
    P = rows if off is None else int(padded_offsets_align(off, align)[-1])
    q_row = np.zeros((rows, cols), np.uint8) if layouts & LAYOUT_ROW else None
    s_row = np.zeros((P, cols // MX_BLOCK), np.uint8) if layouts & LAYOUT_ROW else None
    q_colT = np.zeros((cols, P), np.uint8) if layouts & LAYOUT_COLT else None
    s_col = np.zeros((cols, P // MX_BLOCK), np.uint8) if layouts & LAYOUT_COLT else None
    _load().orc_mx_quantize(_ptr(x), rows, cols, cols, fmt, layouts, _ptr(off), G, int(align), _ptr(q_row),
                            _ptr(s_row), _ptr(q_colT), P, _ptr(s_col))
    return dict(q_row=q_row, s_row=s_row, q_colT=q_colT, s_col=s_col)


def mx_gemm(A, fa, sA, B, fb, sB, points=None):
    """MX GEMM in double: A [M, K] u8 with E8M0 codes sA [M, K/32], B [N, K]
    with sB [N, K/32].  Returns (ref, bound) ([M, N] or [npts])."""
    A = _c(A, np.uint8); B = _c(B, np.uint8)
    sA = _c(sA, np.uint8); sB = _c(sB, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    if points is None:
        ref = np.zeros((M, N)); bound = np.zeros((M, N)); pm = pn = None; npts = 0
    else:
        pm = _c(points[0], np.int64); pn = _c(points[1], np.int64); npts = pm.size
        ref = np.zeros(npts); bound = np.zeros(npts)
    _load().orc_mx_gemm(_ptr(A), fa, K, _ptr(sA), sA.shape[1], _ptr(B), fb, K, _ptr(sB), sB.shape[1], M, N, K,
                        _ptr(pm), _ptr(pn), npts, _ptr(ref), _ptr(bound))
    return ref, bound


# --- MoE prologues: gather (permute) and SwiGLU ------------------------------

def bf16_from_double(x: float) -> int:
    """bf16 bit pattern of x rounded once to the nearest bf16 (ties to even)."""
    return int(_load().orc_bf16_from_double(float(x)))


def swiglu_bf16(g_bits, u_bits) -> np.ndarray:
    """h = bf16_rne(silu(g) * u) element-wise on bf16 bit patterns: the exact
    value (evaluated in double precision) rounded once to bf16."""
    g = _c(g_bits, np.uint16)
    u = _c(u_bits, np.uint16)
    assert g.shape == u.shape
    h = np.zeros(g.shape, np.uint16)
    _load().orc_swiglu_bf16(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def mx_permute_quantize(x_bits, src_rows, fmt, layouts=LAYOUT_ROW | LAYOUT_COLT, offsets=None, align=128):
    """Gather rows x[src_rows] (the permutation of token rows into expert
    order), then MX-quantize them (see mx_quantize)."""
    x = _c(x_bits, np.uint16)
    return mx_quantize(x[np.asarray(src_rows, np.int64)], fmt, layouts, offsets=offsets, align=align)


def mx_swiglu_quantize(gate_up_bits, fmt, layouts=LAYOUT_ROW | LAYOUT_COLT, offsets=None, align=128):
    """h = SwiGLU of a [rows, 2F] gate|up tensor (gate in columns [0, F), up
    in [F, 2F)), then MX quantize of h.  Returns the mx_quantize dict plus h."""
    gu = _c(gate_up_bits, np.uint16)
    F = gu.shape[1] // 2
    h = swiglu_bf16(gu[:, :F], gu[:, F:])
    out = mx_quantize(h, fmt, layouts, offsets=offsets, align=align)
    out["h"] = h
    return out


def permute_quantize(x_bits, src_rows, fmt, kind, offsets, margin=0, layouts=LAYOUT_ROW | LAYOUT_COLT):
    """Gather rows x[src_rows] (routed token rows in expert order), then
    quantize them (see quantize)."""
    x = _c(x_bits, np.uint16)
    return quantize(x[np.asarray(src_rows, np.int64)], fmt, kind, margin=margin, layouts=layouts, offsets=offsets)


def swiglu_quantize(gate_up_bits, fmt, kind, offsets, margin=0, layouts=LAYOUT_ROW | LAYOUT_COLT):
    """h = SwiGLU of a [rows, 2F] gate|up tensor, then quantize h (see
    quantize).  Returns the quantize dict plus h."""
    gu = _c(gate_up_bits, np.uint16)
    F = gu.shape[1] // 2
    h = swiglu_bf16(gu[:, :F], gu[:, F:])
    out = quantize(h, fmt, kind, margin=margin, layouts=layouts, offsets=offsets)
    out["h"] = h
    return out


# --- blockwise (1 x 128 / 128 x 128 blocks, power-of-two scales) -------------

def blockwise_code(amax: float, fmt: int) -> int:
    """E8M0 code of 1/s, s = the largest power of two with amax * s <= fp8_max."""
    return _load().orc_blockwise_code(float(amax), int(fmt))


def blockwise_quantize(x_bits, fmt, block_rows, layouts=LAYOUT_ROW | LAYOUT_COLT):
    """Blockwise quantize (block_rows 1: 1 x 128 activation blocks, 128:
    128 x 128 weight blocks).  Returns q_row, s_row [rows, cols/32], q_colT
    [cols, rows], s_col [cols, rows/32] with per-32-block E8M0 codes."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    q_row = np.zeros((rows, cols), np.uint8) if layouts & LAYOUT_ROW else None
    s_row = np.zeros((rows, cols // 32), np.uint8) if layouts & LAYOUT_ROW else None
    q_colT = np.zeros((cols, rows), np.uint8) if layouts & LAYOUT_COLT else None
    s_col = np.zeros((cols, rows // 32), np.uint8) if layouts & LAYOUT_COLT else None
    _load().orc_blockwise_quantize(_ptr(x), rows, cols, cols, fmt, block_rows, layouts, _ptr(q_row), _ptr(s_row),
                                   _ptr(q_colT), _ptr(s_col))
    return dict(q_row=q_row, s_row=s_row, q_colT=q_colT, s_col=s_col)


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel outer loops (results do not depend on it)."""
    _load().orc_set_threads(int(n))
