"""Host-only checks of the C ABI (no GPU needed, no kernel launched).

  * libfp8gb.so loads and exports every function that include/fp8gb.h
    declares;
  * argument validation rejects bad calls with the documented status before
    anything touches the device;
  * the grouped-layout helper computes the padded offsets.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import fp8_mixed_precision_scale_gb300 as fp8
from fp8_mixed_precision_scale_gb300 import build as fp8build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8gb.h")

OK, INVALID, UNSUPPORTED, ALIGN, CUDA = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    fp8build.build()
    return fp8.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("fp8_quantize", "fp8_update_amax_history", "fp8_scaled_gemm", "fp8_grouped_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fp8.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s+(\w+)", out.stdout))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(fp8.EXPORTED) <= set(declared_functions())


def test_library_has_no_torch_dependency():
    out = subprocess.run(["ldd", fp8.LIB_PATH], capture_output=True, text=True)
    names = [line.split()[0] for line in out.stdout.splitlines() if line.strip()]   # not the load addresses
    assert not any("torch" in n or n.startswith("libc10") for n in names), names


def test_status_strings(lib):
    assert lib.fp8_status_string(0) == b"FP8_OK"
    assert lib.fp8_status_string(5) == b"FP8_ERR_TIMEOUT"
    assert lib.fp8_status_string(99) == b"FP8_ERR_UNKNOWN"
    assert lib.fp8_version().startswith(b"fp8gb")


FAKE = 0x10000  # a 16-byte-aligned non-null address: validation never dereferences it


def q_call(lib, **kw):
    args = dict(x=FAKE, rows=64, cols=64, ld_x=64, fmt=0, kind=0, margin=0, layouts=3, scale_in=FAKE,
                amax_out=FAKE, q_row=FAKE, sinv_row=FAKE, q_colT=FAKE, ld_colT=64, sinv_col=FAKE, offsets=None,
                G=0)
    args.update(kw)
    rec = fp8.fp8_recipe_t(args["kind"], args["margin"], 1024, 0)
    P = ctypes.c_void_p
    return lib.fp8_quantize(P(args["x"]), args["rows"], args["cols"], args["ld_x"], args["fmt"], ctypes.byref(rec),
                            args["layouts"], P(args["scale_in"]), P(args["amax_out"]), P(args["q_row"]),
                            P(args["sinv_row"]), P(args["q_colT"]), args["ld_colT"], P(args["sinv_col"]),
                            P(args["offsets"]), args["G"], None)


def test_quantize_validation(lib):
    assert q_call(lib, x=None) == INVALID
    assert q_call(lib, rows=-1) == INVALID
    assert q_call(lib, cols=0) == INVALID
    assert q_call(lib, ld_x=32) == INVALID
    assert q_call(lib, fmt=4) == INVALID
    assert q_call(lib, fmt=7) == INVALID
    assert q_call(lib, kind=3) == INVALID
    assert q_call(lib, margin=-1) == INVALID
    assert q_call(lib, margin=65) == INVALID
    assert q_call(lib, layouts=0) == INVALID
    assert q_call(lib, layouts=4) == INVALID
    assert q_call(lib, q_row=None) == INVALID
    assert q_call(lib, sinv_col=None) == INVALID
    assert q_call(lib, scale_in=None) == INVALID      # delayed needs the stored scale
    assert q_call(lib, amax_out=None) == INVALID      # ... and the history slot
    assert q_call(lib, kind=1, amax_out=None) == INVALID
    assert q_call(lib, cols=60, ld_x=64) == ALIGN
    assert q_call(lib, ld_x=68) == ALIGN
    assert q_call(lib, x=FAKE + 8) == ALIGN
    assert q_call(lib, ld_colT=72) == ALIGN
    assert q_call(lib, ld_colT=48) == INVALID         # shorter than rows
    assert q_call(lib, offsets=FAKE, G=0) == INVALID
    assert q_call(lib, G=3) == INVALID                # equal groups: 64 rows do not split into 3
    assert q_call(lib, G=2) == INVALID                # equal groups of 32 rows: not a multiple of 64
    assert q_call(lib, G=-1) == INVALID


def r_call(lib, **kw):
    args = dict(x=FAKE, rows=64, cols=64, ld_x=64, fmt=0, margin=0, layouts=3, amax_out=None, q_row=FAKE,
                sinv_row=FAKE, q_colT=FAKE, ld_colT=64, sinv_col=FAKE)
    args.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_quantize_rowwise_resident(P(args["x"]), args["rows"], args["cols"], args["ld_x"], args["fmt"],
                                             args["margin"], args["layouts"], P(args["amax_out"]), P(args["q_row"]),
                                             P(args["sinv_row"]), P(args["q_colT"]), args["ld_colT"],
                                             P(args["sinv_col"]), None)


def test_resident_quantize_validation(lib):
    """The single-launch rowwise quantize checks what fp8_quantize checks for
    a plain rowwise tensor.  An empty tensor passes validation and is
    launched (it writes the column scales and the amax when asked for), so
    without a GPU it gets as far as the CUDA error; the call asks for neither,
    so on a GPU it touches no memory at all."""
    assert r_call(lib, x=None) == INVALID
    assert r_call(lib, rows=-1) == INVALID
    assert r_call(lib, cols=0) == INVALID
    assert r_call(lib, ld_x=32) == INVALID
    assert r_call(lib, fmt=4) == INVALID
    assert r_call(lib, margin=-1) == INVALID
    assert r_call(lib, margin=65) == INVALID
    assert r_call(lib, layouts=0) == INVALID
    assert r_call(lib, layouts=4) == INVALID
    assert r_call(lib, q_row=None) == INVALID
    assert r_call(lib, sinv_row=None) == INVALID
    assert r_call(lib, q_colT=None) == INVALID
    assert r_call(lib, sinv_col=None) == INVALID
    assert r_call(lib, cols=60, ld_x=64) == ALIGN
    assert r_call(lib, ld_x=68) == ALIGN
    assert r_call(lib, x=FAKE + 8) == ALIGN
    assert r_call(lib, q_row=FAKE + 4) == ALIGN
    assert r_call(lib, ld_colT=72) == ALIGN
    assert r_call(lib, ld_colT=48) == INVALID         # shorter than rows
    assert r_call(lib, rows=0, x=None, layouts=1, q_row=None, sinv_row=None, q_colT=None,
                  sinv_col=None) in (OK, CUDA)


def g_call(lib, **kw):
    a = dict(A=FAKE, fa=0, lda=128, B=FAKE, fb=0, ldb=128, M=128, N=256, K=128, sa=FAKE, sam=0, sb=FAKE, sbm=0,
             C=FAKE, ldc=256)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_scaled_gemm(P(a["A"]), a["fa"], a["lda"], P(a["B"]), a["fb"], a["ldb"], a["M"], a["N"], a["K"],
                               P(a["sa"]), a["sam"], P(a["sb"]), a["sbm"], P(a["C"]), a["ldc"], None)


def test_gemm_validation(lib):
    assert g_call(lib, A=None) == INVALID
    assert g_call(lib, C=None) == INVALID
    assert g_call(lib, fa=2) == UNSUPPORTED
    assert g_call(lib, fb=3) == UNSUPPORTED
    assert g_call(lib, fb=5) == INVALID
    assert g_call(lib, M=0) == INVALID
    assert g_call(lib, K=0) == INVALID
    assert g_call(lib, lda=64) == INVALID
    assert g_call(lib, ldc=128) == INVALID
    assert g_call(lib, sam=2) == INVALID
    assert g_call(lib, K=120, lda=128) == ALIGN
    assert g_call(lib, lda=136) == ALIGN
    assert g_call(lib, A=FAKE + 4) == ALIGN
    assert g_call(lib, C=FAKE + 1) == ALIGN


def gg_call(lib, **kw):
    a = dict(mode=0, A=FAKE, fa=0, B=FAKE, fb=0, off=FAKE, G=4, Mt=100, N=256, K=128, sa=FAKE, sam=1, sb=FAKE,
             sbm=1, C=FAKE, ldT=0)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_grouped_gemm(a["mode"], P(a["A"]), a["fa"], P(a["B"]), a["fb"], P(a["off"]), a["G"], a["Mt"],
                                a["N"], a["K"], P(a["sa"]), a["sam"], P(a["sb"]), a["sbm"], P(a["C"]), a["ldT"], None)


def test_grouped_gemm_validation(lib):
    assert gg_call(lib, off=None) == INVALID
    assert gg_call(lib, mode=2) == INVALID
    assert gg_call(lib, G=0) == INVALID
    assert gg_call(lib, G=5000) == INVALID
    assert gg_call(lib, fa=2) == UNSUPPORTED
    assert gg_call(lib, K=120) == ALIGN
    assert gg_call(lib, mode=1, ldT=40) == ALIGN
    assert gg_call(lib, mode=1, ldT=0) == ALIGN


def test_update_validation(lib):
    P = ctypes.c_void_p
    call = lambda **kw: lib.fp8_update_amax_history(  # noqa: E731
        P(kw.get("h", FAKE)), P(FAKE), P(FAKE), P(FAKE), kw.get("n", 4), kw.get("L", 16), kw.get("algo", 0),
        kw.get("margin", 0), None, None)
    assert call(h=None) == INVALID
    assert call(n=0) == INVALID
    assert call(L=0) == INVALID
    assert call(L=40000) == INVALID
    assert call(algo=2) == INVALID
    assert call(margin=70) == INVALID
    assert call(h=FAKE + 2) == ALIGN


def test_padded_offsets_helper(lib):
    total, poff = fp8.fp8_group_padded_offsets([0, 5, 5, 38, 39, 39, 79])
    assert total == 192
    assert list(poff.numpy()) == [0, 32, 32, 96, 128, 128, 192]
    total64, _ = fp8.fp8_group_padded_offsets([0, 5, 5, 38], align=64)
    assert total64 == 128
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_group_padded_offsets([0, 5, 3])
    off = np.array([0, 1], np.int32)
    assert lib.fp8_group_padded_offsets(ctypes.c_void_p(off.ctypes.data), 1, 24, None) == -1


def test_format_roles():
    assert fp8.format_for("e4m3", "grad") == fp8.E4M3FN
    assert fp8.format_for("hybrid", "grad") == fp8.E5M2
    assert fp8.format_for("hybrid", "weight") == fp8.E4M3FN


def test_mx_scale_bytes(lib):
    assert lib.fp8_mx_scale_bytes(5, 5) == 2 * 128 * 4    # ceil(5/4) K tiles x roundup(5,128) rows x 4
    assert lib.fp8_mx_scale_bytes(128, 128) == 32 * 128 * 4
    assert lib.fp8_mx_scale_bytes(129, 4) == 1 * 256 * 4
    assert lib.fp8_mx_scale_bytes(0, 4) == 0
    assert lib.fp8_mx_scale_bytes(-1, 4) == -1


def mxq_call(lib, **kw):
    a = dict(x=FAKE, rows=64, cols=64, ld_x=64, fmt=0, layouts=3, q_row=FAKE, s_row=FAKE, q_colT=FAKE, ld_colT=64,
             s_col=FAKE, off=None, G=0)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_mx_quantize(P(a["x"]), a["rows"], a["cols"], a["ld_x"], a["fmt"], a["layouts"], P(a["q_row"]),
                               P(a["s_row"]), P(a["q_colT"]), a["ld_colT"], P(a["s_col"]), P(a["off"]), a["G"],
                               None)


def test_mx_quantize_validation(lib):
    assert mxq_call(lib, x=None) == INVALID
    assert mxq_call(lib, fmt=2) == UNSUPPORTED
    assert mxq_call(lib, fmt=3) == UNSUPPORTED
    assert mxq_call(lib, fmt=4) == INVALID
    assert mxq_call(lib, layouts=0) == INVALID
    assert mxq_call(lib, q_row=None) == INVALID
    assert mxq_call(lib, s_col=None) == INVALID
    assert mxq_call(lib, cols=48, ld_x=64) == ALIGN        # blocks of 32 along the row
    assert mxq_call(lib, rows=40) == ALIGN                 # transposed layout: blocks of 32 rows
    assert mxq_call(lib, ld_colT=48) == INVALID            # shorter than rows
    assert mxq_call(lib, ld_colT=72) == ALIGN
    assert mxq_call(lib, x=FAKE + 8) == ALIGN
    assert mxq_call(lib, s_row=FAKE + 2) == ALIGN
    assert mxq_call(lib, off=FAKE, G=0) == INVALID
    assert mxq_call(lib, G=2) == INVALID
    assert mxq_call(lib, rows=0, x=None) == OK             # nothing to do


def mxg_call(lib, **kw):
    a = dict(A=FAKE, fa=0, lda=128, sA=FAKE, B=FAKE, fb=0, ldb=128, sB=FAKE, M=128, N=224, K=128, C=FAKE, ldc=224)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_mx_gemm(P(a["A"]), a["fa"], a["lda"], P(a["sA"]), P(a["B"]), a["fb"], a["ldb"], P(a["sB"]),
                           a["M"], a["N"], a["K"], P(a["C"]), a["ldc"], None)


def test_mx_gemm_validation(lib):
    assert mxg_call(lib, sA=None) == INVALID
    assert mxg_call(lib, fa=2) == UNSUPPORTED
    assert mxg_call(lib, fb=6) == INVALID
    assert mxg_call(lib, K=0) == INVALID
    assert mxg_call(lib, K=112) == ALIGN                   # K must be whole 32-element blocks
    assert mxg_call(lib, sB=FAKE + 4) == ALIGN             # scale tiles are bulk copies
    assert mxg_call(lib, lda=136) == ALIGN
    assert mxg_call(lib, ldc=100) == INVALID


def mxgg_call(lib, **kw):
    a = dict(mode=0, A=FAKE, fa=0, sA=FAKE, B=FAKE, fb=0, sB=FAKE, off=FAKE, G=4, Mt=100, N=256, K=128, C=FAKE,
             ldT=0)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.fp8_mx_grouped_gemm(a["mode"], P(a["A"]), a["fa"], P(a["sA"]), P(a["B"]), a["fb"], P(a["sB"]),
                                   P(a["off"]), a["G"], a["Mt"], a["N"], a["K"], P(a["C"]), a["ldT"], None)


def test_mx_grouped_gemm_validation(lib):
    assert mxgg_call(lib, off=None) == INVALID
    assert mxgg_call(lib, mode=2) == INVALID               # transposed B: ld_T shorter than G * kpad
    assert mxgg_call(lib, mode=2, ldT=4 * 128 + 8) == ALIGN
    assert mxgg_call(lib, mode=3) == INVALID
    assert mxgg_call(lib, G=2000) == INVALID
    assert mxgg_call(lib, fa=3) == UNSUPPORTED
    assert mxgg_call(lib, K=96 + 16) == ALIGN
    assert mxgg_call(lib, N=254) == ALIGN                  # scale rows of a tile start on a word boundary
    assert mxgg_call(lib, N=320) == ALIGN                  # M-grouped: experts' scale rows start 128-row blocks
    assert mxgg_call(lib, mode=1, ldT=192) == ALIGN        # groups padded to 128 columns
    assert mxgg_call(lib, mode=1, ldT=256, K=130) == ALIGN


def test_mx_fused_validation(lib):
    P = ctypes.c_void_p
    perm = lambda **kw: lib.fp8_mx_permute_quantize(  # noqa: E731
        P(kw.get("x", FAKE)), kw.get("x_rows", 64), kw.get("cols", 64), 64, P(kw.get("src", FAKE)),
        kw.get("rows", 64), kw.get("fmt", 0), 1, P(FAKE), P(FAKE), None, 0, None, None, 0, None)
    assert perm(src=None) == INVALID
    assert perm(x_rows=0) == INVALID
    assert perm(cols=48) == ALIGN                          # 48 columns are not whole 32-element blocks
    assert perm(fmt=2) == UNSUPPORTED
    assert perm(rows=0, src=None) == OK
    swi = lambda **kw: lib.fp8_mx_swiglu_quantize(  # noqa: E731
        P(FAKE), 64, kw.get("F", 64), kw.get("ld", 128), 0, 1, P(kw.get("h", None)), kw.get("ld_h", 0),
        P(FAKE), P(FAKE), None, 0, None, None, 0, None)
    assert swi(ld=100) == INVALID                          # shorter than 2F
    assert swi(F=48, ld=96) == ALIGN
    assert swi(h=FAKE, ld_h=32) == INVALID
    assert swi(h=FAKE + 8, ld_h=64) == ALIGN


def test_blockwise_validation(lib):
    P = ctypes.c_void_p
    bw = lambda **kw: lib.fp8_blockwise_quantize(  # noqa: E731
        P(kw.get("x", FAKE)), kw.get("rows", 128), kw.get("cols", 128), kw.get("ld", 128), kw.get("fmt", 0),
        kw.get("br", 1), kw.get("lay", 3), P(FAKE), P(FAKE), P(FAKE), kw.get("ldT", 128), P(FAKE), None)
    assert bw(br=64) == INVALID
    assert bw(fmt=2) == UNSUPPORTED
    assert bw(cols=96, ld=128) == ALIGN                     # whole 128-column blocks
    assert bw(rows=96, ldT=128) == ALIGN                    # transposed layout: whole 128-row blocks
    assert bw(rows=96, lay=1, br=128) == ALIGN              # weights: 128 x 128 blocks
    assert bw(ldT=136) == ALIGN                            # not a multiple of 16
    assert bw(rows=256, ldT=128) == INVALID                 # ld_colT shorter than rows
