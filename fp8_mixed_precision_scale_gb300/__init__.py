"""Python binding of the GB300 FP8 linear-layer library (libfp8gb.so).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  If the
library is missing, every entry point raises -- there is no fallback.

The C ABI (include/fp8gb.h) is mirrored one to one:

  fp8_quantize             fused amax + scale + saturating cast, rowwise and
                           colwise-transposed layouts from one read
  fp8_update_amax_history  delayed-scaling history roll + scale update
  fp8_scaled_gemm          FP8 x FP8 -> bf16 with scales in the epilogue
  fp8_grouped_gemm         the same over MoE expert groups
  fp8_group_padded_offsets host helper for the grouped colwise layout
  fp8_sync_status          stream sync + device error word

`quantize`, `scaled_gemm`, `grouped_gemm` are convenience wrappers that
allocate the outputs with torch and call the entry points above.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

E4M3FN, E5M2, E4M3FNUZ, E5M2FNUZ = 0, 1, 2, 3
DELAYED, TENSORWISE, ROWWISE = 0, 1, 2
MOST_RECENT, MAX = 0, 1
LAYOUT_ROW, LAYOUT_COLT = 1, 2
SCALE_TENSOR, SCALE_PER_ROW = 0, 1
GROUPED_M, GROUPED_K, GROUPED_M_BT = 0, 1, 2
STATUS = {0: "FP8_OK", 1: "FP8_ERR_INVALID_ARG", 2: "FP8_ERR_UNSUPPORTED", 3: "FP8_ERR_ALIGNMENT",
          4: "FP8_ERR_CUDA", 5: "FP8_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8gb.so")
EXPORTED = ("fp8_quantize", "fp8_update_amax_history", "fp8_scaled_gemm", "fp8_grouped_gemm",
            "fp8_group_padded_offsets", "fp8_sync_status", "fp8_selftest_bounded_wait", "fp8_status_string",
            "fp8_last_cuda_error", "fp8_version", "fp8_mx_scale_bytes", "fp8_mx_quantize", "fp8_mx_gemm",
            "fp8_mx_grouped_gemm", "fp8_mx_permute_quantize", "fp8_mx_swiglu_quantize", "fp8_blockwise_quantize",
            "fp8_quantize_rowwise_resident", "fp8_permute_quantize", "fp8_swiglu_quantize")
MX_BLOCK = 32
MX_GROUP_ALIGN = 128

_lock = threading.Lock()
_lib = None


class Fp8Error(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class fp8_recipe_t(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("margin", ctypes.c_int), ("history_len", ctypes.c_int),
                ("algo", ctypes.c_int)]


@dataclass
class Recipe:
    """The recipe knobs: kind (DELAYED / TENSORWISE / ROWWISE), margin,
    history_len, algo (MOST_RECENT / MAX)."""
    kind: int = DELAYED
    margin: int = 0
    history_len: int = 1024
    algo: int = MOST_RECENT

    def c(self) -> fp8_recipe_t:
        return fp8_recipe_t(self.kind, self.margin, self.history_len, self.algo)


def format_for(fp8: str, role: str) -> int:
    """FP8 format of a tensor role under the "e4m3" or "hybrid" setting:
    hybrid keeps activations and weights in E4M3 and gradients in E5M2."""
    if fp8 == "e4m3":
        return E4M3FN
    if fp8 == "hybrid":
        return E5M2 if role in ("grad", "grad_output", "dy") else E4M3FN
    raise ValueError(f"unknown fp8 setting {fp8!r}")


def load_library():
    """Load libfp8gb.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with fp8_mixed_precision_scale_gb300.build")
            lib = ctypes.CDLL(LIB_PATH)
            P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.fp8_quantize.restype = i32
            lib.fp8_quantize.argtypes = [P, i64, i64, i64, i32, ctypes.POINTER(fp8_recipe_t), i32, P, P, P, P, P,
                                         i64, P, P, i32, P]
            lib.fp8_quantize_rowwise_resident.restype = i32
            lib.fp8_quantize_rowwise_resident.argtypes = [P, i64, i64, i64, i32, i32, i32, P, P, P, P, i64, P, P]
            lib.fp8_permute_quantize.restype = i32
            lib.fp8_permute_quantize.argtypes = [P, i64, i64, i64, P, i64, i32, i32, i32, P, P, P, P, i64, P, P, i32,
                                                 P]
            lib.fp8_swiglu_quantize.restype = i32
            lib.fp8_swiglu_quantize.argtypes = [P, i64, i64, i64, i32, i32, i32, P, i64, P, P, P, P, i64, P, P, i32, P]
            lib.fp8_update_amax_history.restype = i32
            lib.fp8_update_amax_history.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P]
            lib.fp8_scaled_gemm.restype = i32
            lib.fp8_scaled_gemm.argtypes = [P, i32, i64, P, i32, i64, i64, i64, i64, P, i32, P, i32, P, i64, P]
            lib.fp8_grouped_gemm.restype = i32
            lib.fp8_grouped_gemm.argtypes = [i32, P, i32, P, i32, P, i32, i64, i64, i64, P, i32, P, i32, P, i64, P]
            lib.fp8_group_padded_offsets.restype = i64
            lib.fp8_group_padded_offsets.argtypes = [P, i32, i32, P]
            lib.fp8_sync_status.restype = i32
            lib.fp8_sync_status.argtypes = [P]
            lib.fp8_selftest_bounded_wait.restype = i32
            lib.fp8_selftest_bounded_wait.argtypes = [i64, P]
            lib.fp8_status_string.restype = ctypes.c_char_p
            lib.fp8_status_string.argtypes = [i32]
            lib.fp8_last_cuda_error.restype = ctypes.c_char_p
            lib.fp8_last_cuda_error.argtypes = []
            lib.fp8_version.restype = ctypes.c_char_p
            lib.fp8_version.argtypes = []
            lib.fp8_mx_scale_bytes.restype = i64
            lib.fp8_mx_scale_bytes.argtypes = [i64, i64]
            lib.fp8_mx_quantize.restype = i32
            lib.fp8_mx_quantize.argtypes = [P, i64, i64, i64, i32, i32, P, P, P, i64, P, P, i32, P]
            lib.fp8_mx_permute_quantize.restype = i32
            lib.fp8_mx_permute_quantize.argtypes = [P, i64, i64, i64, P, i64, i32, i32, P, P, P, i64, P, P, i32, P]
            lib.fp8_mx_swiglu_quantize.restype = i32
            lib.fp8_mx_swiglu_quantize.argtypes = [P, i64, i64, i64, i32, i32, P, i64, P, P, P, i64, P, P, i32, P]
            lib.fp8_blockwise_quantize.restype = i32
            lib.fp8_blockwise_quantize.argtypes = [P, i64, i64, i64, i32, i32, i32, P, P, P, i64, P, P]
            lib.fp8_mx_gemm.restype = i32
            lib.fp8_mx_gemm.argtypes = [P, i32, i64, P, P, i32, i64, P, i64, i64, i64, P, i64, P]
            lib.fp8_mx_grouped_gemm.restype = i32
            lib.fp8_mx_grouped_gemm.argtypes = [i32, P, i32, P, P, i32, P, P, i32, i64, i64, i64, P, i64, P]
            _lib = lib
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str):
    if status != 0:
        detail = load_library().fp8_last_cuda_error().decode() if status == 4 else ""
        raise Fp8Error(status, where, detail)


# --- the C entry points ------------------------------------------------------

def fp8_quantize(x, rows, cols, ld_x, fmt, recipe: Recipe, layouts, scale_in, amax_out, q_row, scale_inv_row,
                 q_colT, ld_colT, scale_inv_col, group_offsets=None, num_groups=0, stream=None, check=True):
    rc = load_library().fp8_quantize(_p(x), rows, cols, ld_x, fmt, ctypes.byref(recipe.c()), layouts,
                                     _p(scale_in), _p(amax_out), _p(q_row), _p(scale_inv_row), _p(q_colT),
                                     ld_colT, _p(scale_inv_col), _p(group_offsets), num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_quantize")
    return rc


def fp8_update_amax_history(hist, scale, scale_inv, fmt, n, L, algo, margin, nonfinite_count=None, stream=None,
                            check=True):
    rc = load_library().fp8_update_amax_history(_p(hist), _p(scale), _p(scale_inv), _p(fmt), n, L, algo, margin,
                                                _p(nonfinite_count), _stream(stream))
    if check:
        _check(rc, "fp8_update_amax_history")
    return rc


def fp8_scaled_gemm(A, fa, lda, B, fb, ldb, M, N, K, sa, sa_mode, sb, sb_mode, C, ldc, stream=None, check=True):
    rc = load_library().fp8_scaled_gemm(_p(A), fa, lda, _p(B), fb, ldb, M, N, K, _p(sa), sa_mode, _p(sb), sb_mode,
                                        _p(C), ldc, _stream(stream))
    if check:
        _check(rc, "fp8_scaled_gemm")
    return rc


def fp8_grouped_gemm(mode, A, fa, B, fb, group_offsets, G, M_total, N, K, sa, sa_mode, sb, sb_mode, C, ld_T=0,
                     stream=None, check=True):
    rc = load_library().fp8_grouped_gemm(mode, _p(A), fa, _p(B), fb, _p(group_offsets), G, M_total, N, K, _p(sa),
                                         sa_mode, _p(sb), sb_mode, _p(C), ld_T, _stream(stream))
    if check:
        _check(rc, "fp8_grouped_gemm")
    return rc


def fp8_group_padded_offsets(host_offsets, align: int = 32):
    """int32 CPU offsets [G+1] -> (total, int64 CPU padded offsets [G+1])."""
    off = torch.as_tensor(host_offsets, dtype=torch.int32).contiguous().cpu()
    G = off.numel() - 1
    out = torch.zeros(G + 1, dtype=torch.int64)
    total = load_library().fp8_group_padded_offsets(_p(off), G, align, _p(out))
    if total < 0:
        raise Fp8Error(1, "fp8_group_padded_offsets")
    return int(total), out


def fp8_mx_scale_bytes(scale_rows: int, blocks: int) -> int:
    return int(load_library().fp8_mx_scale_bytes(scale_rows, blocks))


def fp8_mx_quantize(x, rows, cols, ld_x, fmt, layouts, q_row, s_row, q_colT, ld_colT, s_col, group_offsets=None,
                    num_groups=0, stream=None, check=True):
    rc = load_library().fp8_mx_quantize(_p(x), rows, cols, ld_x, fmt, layouts, _p(q_row), _p(s_row), _p(q_colT),
                                        ld_colT, _p(s_col), _p(group_offsets), num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_mx_quantize")
    return rc


def fp8_mx_permute_quantize(x, x_rows, cols, ld_x, src_rows, rows, fmt, layouts, q_row, s_row, q_colT, ld_colT,
                            s_col, group_offsets=None, num_groups=0, stream=None, check=True):
    rc = load_library().fp8_mx_permute_quantize(_p(x), x_rows, cols, ld_x, _p(src_rows), rows, fmt, layouts,
                                                _p(q_row), _p(s_row), _p(q_colT), ld_colT, _p(s_col),
                                                _p(group_offsets), num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_mx_permute_quantize")
    return rc


def fp8_mx_swiglu_quantize(gate_up, rows, F, ld, fmt, layouts, h, ld_h, q_row, s_row, q_colT, ld_colT, s_col,
                           group_offsets=None, num_groups=0, stream=None, check=True):
    rc = load_library().fp8_mx_swiglu_quantize(_p(gate_up), rows, F, ld, fmt, layouts, _p(h), ld_h, _p(q_row),
                                               _p(s_row), _p(q_colT), ld_colT, _p(s_col), _p(group_offsets),
                                               num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_mx_swiglu_quantize")
    return rc


def fp8_quantize_rowwise_resident(x, rows, cols, ld_x, fmt, margin, layouts, amax_out, q_row, scale_inv_row, q_colT,
                                  ld_colT, scale_inv_col, stream=None, check=True):
    rc = load_library().fp8_quantize_rowwise_resident(_p(x), rows, cols, ld_x, fmt, margin, layouts, _p(amax_out),
                                                      _p(q_row), _p(scale_inv_row), _p(q_colT), ld_colT,
                                                      _p(scale_inv_col), _stream(stream))
    if check:
        _check(rc, "fp8_quantize_rowwise_resident")
    return rc


def fp8_permute_quantize(x, x_rows, cols, ld_x, src_rows, rows, fmt, margin, layouts, amax_out, q_row,
                         scale_inv_row, q_colT, ld_colT, scale_inv_col, group_offsets, num_groups, stream=None,
                         check=True):
    rc = load_library().fp8_permute_quantize(_p(x), x_rows, cols, ld_x, _p(src_rows), rows, fmt, margin, layouts,
                                             _p(amax_out), _p(q_row), _p(scale_inv_row), _p(q_colT), ld_colT,
                                             _p(scale_inv_col), _p(group_offsets), num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_permute_quantize")
    return rc


def fp8_swiglu_quantize(gate_up, rows, F, ld, fmt, margin, layouts, h, ld_h, amax_out, q_row, scale_inv_row,
                        q_colT, ld_colT, scale_inv_col, group_offsets, num_groups, stream=None, check=True):
    rc = load_library().fp8_swiglu_quantize(_p(gate_up), rows, F, ld, fmt, margin, layouts, _p(h), ld_h,
                                            _p(amax_out), _p(q_row), _p(scale_inv_row), _p(q_colT), ld_colT,
                                            _p(scale_inv_col), _p(group_offsets), num_groups, _stream(stream))
    if check:
        _check(rc, "fp8_swiglu_quantize")
    return rc


def fp8_blockwise_quantize(x, rows, cols, ld_x, fmt, block_rows, layouts, q_row, s_row, q_colT, ld_colT, s_col,
                           stream=None, check=True):
    rc = load_library().fp8_blockwise_quantize(_p(x), rows, cols, ld_x, fmt, block_rows, layouts, _p(q_row),
                                               _p(s_row), _p(q_colT), ld_colT, _p(s_col), _stream(stream))
    if check:
        _check(rc, "fp8_blockwise_quantize")
    return rc


def fp8_mx_gemm(A, fa, lda, sA, B, fb, ldb, sB, M, N, K, C, ldc, stream=None, check=True):
    rc = load_library().fp8_mx_gemm(_p(A), fa, lda, _p(sA), _p(B), fb, ldb, _p(sB), M, N, K, _p(C), ldc,
                                    _stream(stream))
    if check:
        _check(rc, "fp8_mx_gemm")
    return rc


def fp8_mx_grouped_gemm(mode, A, fa, sA, B, fb, sB, group_offsets, G, M_total, N, K, C, ld_T=0, stream=None,
                        check=True):
    rc = load_library().fp8_mx_grouped_gemm(mode, _p(A), fa, _p(sA), _p(B), fb, _p(sB), _p(group_offsets), G,
                                            M_total, N, K, _p(C), ld_T, _stream(stream))
    if check:
        _check(rc, "fp8_mx_grouped_gemm")
    return rc


def fp8_sync_status(stream=None) -> int:
    return load_library().fp8_sync_status(_stream(stream))


def fp8_selftest_bounded_wait(wait_ns: int, stream=None) -> int:
    return load_library().fp8_selftest_bounded_wait(int(wait_ns), _stream(stream))


def version() -> str:
    return load_library().fp8_version().decode()


# --- convenience wrappers (allocate outputs with torch) -----------------------

@dataclass
class Quantized:
    q_row: torch.Tensor | None
    scale_inv_row: torch.Tensor | None
    q_colT: torch.Tensor | None
    scale_inv_col: torch.Tensor | None
    ld_colT: int


def quantize(x: torch.Tensor, fmt: int, recipe: Recipe, layouts: int = LAYOUT_ROW | LAYOUT_COLT, scale_in=None,
             amax_out=None, group_offsets=None, host_offsets=None, stream=None, equal_groups: int = 0) -> Quantized:
    """Quantize a CUDA bf16 [rows, cols] tensor (row stride x.stride(0)).

    Grouped (MoE) tensors pass the device offsets and their CPU copy
    (host_offsets) so the padded colwise width can be sized here; a stack of
    equal groups (expert weights) may pass equal_groups = the number of
    groups instead (rows / equal_groups a multiple of 64).
    """
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = x.device
    G = 0
    if group_offsets is not None:
        G = group_offsets.numel() - 1
        ld_colT, _ = fp8_group_padded_offsets(host_offsets)
        ld_colT = max(16, (ld_colT + 15) // 16 * 16)
    else:
        G = equal_groups
        ld_colT = max(16, (rows + 15) // 16 * 16)
    q_row = sr = q_colT = sc = None
    if layouts & LAYOUT_ROW:
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        sr = torch.empty(rows if recipe.kind == ROWWISE else 1, dtype=torch.float32, device=dev)
    if layouts & LAYOUT_COLT:
        q_colT = torch.empty((cols, ld_colT), dtype=torch.uint8, device=dev)
        nsc = (cols * (G if G else 1)) if recipe.kind == ROWWISE else 1
        sc = torch.empty(nsc, dtype=torch.float32, device=dev)
    fp8_quantize(x, rows, cols, x.stride(0), fmt, recipe, layouts, scale_in, amax_out, q_row, sr, q_colT, ld_colT,
                 sc, group_offsets, G, stream)
    return Quantized(q_row, sr, q_colT, sc, ld_colT)


def quantize_rowwise_resident(x: torch.Tensor, fmt: int, margin: int = 0, layouts: int = LAYOUT_ROW | LAYOUT_COLT,
                              amax_out=None, stream=None) -> Quantized:
    """The rowwise recipe of quantize() for a plain CUDA bf16 [rows, cols]
    tensor in one cooperative launch (same results; fewer launches, and the
    second read of x comes from L2)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = x.device
    ld_colT = max(16, (rows + 15) // 16 * 16)
    q_row = sr = q_colT = sc = None
    if layouts & LAYOUT_ROW:
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        sr = torch.empty(max(rows, 1), dtype=torch.float32, device=dev)
    if layouts & LAYOUT_COLT:
        q_colT = torch.empty((cols, ld_colT), dtype=torch.uint8, device=dev)
        sc = torch.empty(cols, dtype=torch.float32, device=dev)
    fp8_quantize_rowwise_resident(x, rows, cols, x.stride(0), fmt, margin, layouts, amax_out, q_row, sr, q_colT,
                                  ld_colT, sc, stream)
    return Quantized(q_row, sr, q_colT, sc, ld_colT)


def _rowwise_outputs(rows, cols, dev, layouts, host_offsets):
    G = len(host_offsets) - 1
    ld_colT, _ = fp8_group_padded_offsets(host_offsets)
    ld_colT = max(16, (ld_colT + 15) // 16 * 16)
    q_row = sr = q_colT = sc = None
    if layouts & LAYOUT_ROW:
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        sr = torch.empty(max(rows, 1), dtype=torch.float32, device=dev)
    if layouts & LAYOUT_COLT:
        q_colT = torch.empty((cols, ld_colT), dtype=torch.uint8, device=dev)
        sc = torch.empty(cols * G, dtype=torch.float32, device=dev)
    return Quantized(q_row, sr, q_colT, sc, ld_colT)


def permute_quantize(x: torch.Tensor, src_rows: torch.Tensor, fmt: int, group_offsets, host_offsets,
                     layouts: int = LAYOUT_ROW | LAYOUT_COLT, margin: int = 0, amax_out=None,
                     stream=None) -> Quantized:
    """Gather x[src_rows] (routed token rows in expert order) and quantize it
    with the rowwise recipe, per-expert column scales, in one pass."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1 and src_rows.dtype == torch.int32
    rows, cols = src_rows.numel(), x.shape[1]
    q = _rowwise_outputs(rows, cols, x.device, layouts, host_offsets)
    fp8_permute_quantize(x, x.shape[0], cols, x.stride(0), src_rows, rows, fmt, margin, layouts, amax_out, q.q_row,
                         q.scale_inv_row, q.q_colT, q.ld_colT, q.scale_inv_col, group_offsets,
                         group_offsets.numel() - 1, stream)
    return q


def swiglu_quantize(gate_up: torch.Tensor, fmt: int, group_offsets, host_offsets,
                    layouts: int = LAYOUT_ROW | LAYOUT_COLT, h_out=None, margin: int = 0, amax_out=None,
                    stream=None) -> Quantized:
    """h = bf16(silu(gate) * up) of a [rows, 2F] gate|up tensor, quantized
    with the rowwise recipe, per-expert column scales, in one pass (h also
    written to h_out when given)."""
    assert gate_up.dtype == torch.bfloat16 and gate_up.dim() == 2 and gate_up.stride(1) == 1
    rows, F = gate_up.shape[0], gate_up.shape[1] // 2
    q = _rowwise_outputs(rows, F, gate_up.device, layouts, host_offsets)
    fp8_swiglu_quantize(gate_up, rows, F, gate_up.stride(0), fmt, margin, layouts, h_out,
                        h_out.stride(0) if h_out is not None else 0, amax_out, q.q_row, q.scale_inv_row, q.q_colT,
                        q.ld_colT, q.scale_inv_col, group_offsets, group_offsets.numel() - 1, stream)
    return q


def scaled_gemm(A: torch.Tensor, fa: int, B: torch.Tensor, fb: int, sa: torch.Tensor, sb: torch.Tensor, K=None,
                out=None, stream=None) -> torch.Tensor:
    """C = bf16(A[:, :K] . B[:, :K]^T * sa * sb); sa/sb of size 1 are per-tensor."""
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    C = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    fp8_scaled_gemm(A, fa, A.stride(0), B, fb, B.stride(0), M, N, K, sa, int(sa.numel() > 1), sb,
                    int(sb.numel() > 1), C, C.stride(0), stream)
    return C


def grouped_gemm(mode: int, A, fa, B, fb, group_offsets, M_total, N, K, sa, sb, ld_T=0, out=None, stream=None):
    G = group_offsets.numel() - 1
    if out is None:
        shape = (G, N, K) if mode == GROUPED_K else (M_total, N)
        out = torch.empty(shape, dtype=torch.bfloat16, device=A.device)
    fp8_grouped_gemm(mode, A, fa, B, fb, group_offsets, G, M_total, N, K, sa, int(sa.numel() > 1), sb,
                     int(sb.numel() > 1), out, ld_T, stream)
    return out


@dataclass
class MxQuantized:
    q_row: torch.Tensor | None     # [rows, cols] u8
    s_row: torch.Tensor | None     # MX scale layout, R = rows (grouped: padded total)
    q_colT: torch.Tensor | None    # [cols, ld_colT] u8
    s_col: torch.Tensor | None     # MX scale layout, R = cols, KB = ld_colT / 32
    ld_colT: int
    scale_rows: int                # R of s_row


def mx_quantize(x: torch.Tensor, fmt: int, layouts: int = LAYOUT_ROW | LAYOUT_COLT, group_offsets=None,
                host_offsets=None, stream=None) -> MxQuantized:
    """MX quantize of a CUDA bf16 [rows, cols] tensor (cols % 32 == 0).

    Grouped (MoE) tensors pass the device offsets and their CPU copy; every
    group is padded to MX_GROUP_ALIGN rows in the padded layouts.
    """
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = x.device
    G = 0
    if group_offsets is not None:
        G = group_offsets.numel() - 1
        P, _ = fp8_group_padded_offsets(host_offsets, MX_GROUP_ALIGN)
    else:
        P = rows
    ld_colT = max(16, (P + 15) // 16 * 16)
    def buf(n):  # never a zero-byte (null) allocation
        return torch.empty(max(16, n), dtype=torch.uint8, device=dev)

    q_row = s_row = q_colT = s_col = None
    if layouts & LAYOUT_ROW:
        q_row = buf(rows * cols)[:rows * cols].view(rows, cols)
        s_row = buf(fp8_mx_scale_bytes(P, cols // MX_BLOCK))
    if layouts & LAYOUT_COLT:
        q_colT = buf(cols * ld_colT)[:cols * ld_colT].view(cols, ld_colT)
        s_col = buf(fp8_mx_scale_bytes(cols, P // MX_BLOCK))
    fp8_mx_quantize(x, rows, cols, x.stride(0), fmt, layouts, q_row, s_row, q_colT, ld_colT, s_col, group_offsets,
                    G, stream)
    return MxQuantized(q_row, s_row, q_colT, s_col, ld_colT, P)


def _mx_outputs(rows, cols, dev, layouts, host_offsets):
    P = fp8_group_padded_offsets(host_offsets, MX_GROUP_ALIGN)[0] if host_offsets is not None else rows
    ld_colT = max(16, (P + 15) // 16 * 16)

    def buf(n):  # never a zero-byte (null) allocation
        return torch.empty(max(16, n), dtype=torch.uint8, device=dev)

    q_row = s_row = q_colT = s_col = None
    if layouts & LAYOUT_ROW:
        q_row = buf(rows * cols)[:rows * cols].view(rows, cols)
        s_row = buf(fp8_mx_scale_bytes(P, cols // MX_BLOCK))
    if layouts & LAYOUT_COLT:
        q_colT = buf(cols * ld_colT)[:cols * ld_colT].view(cols, ld_colT)
        s_col = buf(fp8_mx_scale_bytes(cols, P // MX_BLOCK))
    return MxQuantized(q_row, s_row, q_colT, s_col, ld_colT, P)


def mx_permute_quantize(x: torch.Tensor, src_rows: torch.Tensor, fmt: int, layouts: int = LAYOUT_ROW | LAYOUT_COLT,
                        group_offsets=None, host_offsets=None, stream=None) -> MxQuantized:
    """Gather x[src_rows] (routed token rows in expert order) and MX-quantize
    them in one pass."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1 and src_rows.dtype == torch.int32
    rows, cols = src_rows.numel(), x.shape[1]
    q = _mx_outputs(rows, cols, x.device, layouts, host_offsets)
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    fp8_mx_permute_quantize(x, x.shape[0], cols, x.stride(0), src_rows, rows, fmt, layouts, q.q_row, q.s_row,
                            q.q_colT, q.ld_colT, q.s_col, group_offsets, G, stream)
    return q


def mx_swiglu_quantize(gate_up: torch.Tensor, fmt: int, layouts: int = LAYOUT_ROW | LAYOUT_COLT, h_out=None,
                       group_offsets=None, host_offsets=None, stream=None) -> MxQuantized:
    """h = bf16(silu(gate) * up) of a [rows, 2F] gate|up tensor, MX-quantized
    in one pass (h also written to h_out when given)."""
    assert gate_up.dtype == torch.bfloat16 and gate_up.dim() == 2 and gate_up.stride(1) == 1
    rows, F = gate_up.shape[0], gate_up.shape[1] // 2
    q = _mx_outputs(rows, F, gate_up.device, layouts, host_offsets)
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    fp8_mx_swiglu_quantize(gate_up, rows, F, gate_up.stride(0), fmt, layouts, h_out,
                           h_out.stride(0) if h_out is not None else 0, q.q_row, q.s_row, q.q_colT, q.ld_colT,
                           q.s_col, group_offsets, G, stream)
    return q


def mx_gemm(A: torch.Tensor, fa: int, sA: torch.Tensor, B: torch.Tensor, fb: int, sB: torch.Tensor, K=None,
            out=None, stream=None) -> torch.Tensor:
    """C = bf16(MX-scaled A[:, :K] . B[:, :K]^T)."""
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    C = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    fp8_mx_gemm(A, fa, A.stride(0), sA, B, fb, B.stride(0), sB, M, N, K, C, C.stride(0), stream)
    return C


def mx_grouped_gemm(mode: int, A, fa, sA, B, fb, sB, group_offsets, M_total, N, K, ld_T=0, out=None, stream=None):
    G = group_offsets.numel() - 1
    if out is None:
        shape = (G, N, K) if mode == GROUPED_K else (M_total, N)
        out = torch.empty(shape, dtype=torch.bfloat16, device=A.device)
    fp8_mx_grouped_gemm(mode, A, fa, sA, B, fb, sB, group_offsets, G, M_total, N, K, out, ld_T, stream)
    return out


def blockwise_quantize(x: torch.Tensor, fmt: int, block_rows: int, layouts: int = LAYOUT_ROW | LAYOUT_COLT,
                       stream=None) -> MxQuantized:
    """Blockwise quantize of a CUDA bf16 [rows, cols] tensor: block_rows 1 for
    activations / gradients (1 x 128 blocks), 128 for weights (128 x 128).
    The scales are in the MX scale layout, ready for mx_gemm."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    q = _mx_outputs(rows, cols, x.device, layouts, None)
    fp8_blockwise_quantize(x, rows, cols, x.stride(0), fmt, block_rows, layouts, q.q_row, q.s_row, q.q_colT,
                           q.ld_colT, q.s_col, stream)
    return q
