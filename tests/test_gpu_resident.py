"""GPU parity of fp8_quantize_rowwise_resident (the rowwise recipe in one
cooperative launch) against the oracle, its argument checks and calls on two
streams.  Its comparison with fp8_quantize's two-pass path (two calls in a
row, every barrier counter reused, the empty tensor) is in
test_zz_no_alloc.py."""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
from parity import assert_codes_equal, assert_f32_bits_equal, bits
from test_gpu_quantize import gen_x

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    fp8.load_library()


def run_resident(x, fmt, layouts=3, margin=0):
    amax = torch.tensor([123.0], dtype=torch.float32, device=DEV)   # overwritten by the call
    q = fp8.quantize_rowwise_resident(x.to(DEV), fmt, margin, layouts, amax_out=amax)
    assert fp8.fp8_sync_status() == 0
    return q, float(amax.cpu()[0])


def check(orc, x, fmt, layouts=3, margin=0, what=""):
    q, amax = run_resident(x, fmt, layouts, margin)
    ref = orc.quantize(bits(x), fmt, orc.ROWWISE, margin=margin, layouts=layouts)
    rows = x.shape[0]
    if layouts & 1:
        assert_codes_equal(q.q_row.cpu().numpy(), ref["q_row"], fmt, what + " q_row")
        assert_f32_bits_equal(q.scale_inv_row.cpu().numpy()[:rows], ref["scale_inv_row"], what + " sinv_row")
    if layouts & 2:
        assert_codes_equal(q.q_colT.cpu().numpy()[:, :rows], ref["q_colT"], fmt, what + " q_colT")
        assert_f32_bits_equal(q.scale_inv_col.cpu().numpy(), ref["scale_inv_col"], what + " sinv_col")
    assert_f32_bits_equal(np.array([amax], np.float32), np.array([ref["amax"]], np.float32), what + " amax")


SHAPES = [(1, 8), (37, 136), (64, 128), (129, 256), (300, 520), (1000, 1032), (2048, 4104)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [0, 1, 2, 3])
def test_resident_matches_oracle(orc, shape, fmt):
    x = gen_x(shape, seed=shape[0] + 3 * shape[1] + fmt, scale=0.3 if fmt in (0, 2) else 1e-3)
    check(orc, x, fmt, what=f"{shape} f{fmt}")


@pytest.mark.parametrize("layouts", [1, 2])
@pytest.mark.parametrize("margin", [0, 3])
def test_resident_single_layout_and_margin(orc, layouts, margin):
    x = gen_x((300, 264), seed=11 + layouts + margin)
    check(orc, x, 0, layouts=layouts, margin=margin, what=f"layouts {layouts} margin {margin}")


def test_resident_special_values(orc):
    """NaN / Inf / zero rows and columns: scales of 1 for zero and non-finite
    amaxes, NaN propagation into the amax, as in the oracle."""
    x = gen_x((200, 136), seed=5)
    x[3, :] = 0
    x[:, 7] = 0
    x[10, 20] = float("inf")
    x[50, 9] = float("nan")
    x[77, :] = 1e-40
    check(orc, x, 1, what="specials")


def test_resident_rejects_bad_arguments():
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((64, 64), dtype=torch.uint8, device=DEV)
    s = torch.empty(64, dtype=torch.float32, device=DEV)
    bad = [
        dict(fmt=7), dict(margin=-1), dict(layouts=0), dict(cols=60),
    ]
    for b in bad:
        args = dict(fmt=0, margin=0, layouts=1, cols=64)
        args.update(b)
        rc = fp8.fp8_quantize_rowwise_resident(x, 64, args["cols"], 64, args["fmt"], args["margin"],
                                               args["layouts"], None, q, s, None, 0, None, check=False)
        assert rc in (1, 3), (b, rc)   # FP8_ERR_INVALID_ARG, FP8_ERR_ALIGNMENT
    rc = fp8.fp8_quantize_rowwise_resident(x, 0, 64, 64, 0, 0, 1, None, None, None, None, 0, None, check=False)
    assert rc == 0


def test_resident_calls_on_two_streams():
    """Calls on two streams, issued back to back without synchronising: each
    takes its own barrier counter, and every result equals the two-pass
    path's."""
    xs = [gen_x((1000, 1032), seed=s).to(DEV) for s in (21, 22)]
    rec = fp8.Recipe(kind=fp8.ROWWISE)
    refs = [fp8.quantize(x, 1, rec, 3) for x in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for _ in range(4):
        for i, (x, st) in enumerate(zip(xs, streams)):
            with torch.cuda.stream(st):
                outs.append((i, fp8.quantize_rowwise_resident(x, 1, stream=st)))
    torch.cuda.synchronize()
    assert fp8.fp8_sync_status() == 0
    for i, q in outs:
        ref = refs[i]
        assert torch.equal(q.q_row, ref.q_row)
        assert torch.equal(q.q_colT[:, :1000], ref.q_colT[:, :1000])
        assert torch.equal(q.scale_inv_row[:1000].view(torch.int32), ref.scale_inv_row.view(torch.int32))
        assert torch.equal(q.scale_inv_col.view(torch.int32), ref.scale_inv_col.view(torch.int32))
