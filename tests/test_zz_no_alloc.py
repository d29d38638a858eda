"""GPU tests of fp8_quantize_rowwise_resident, the entry point that allocates
nothing: its barrier counters sit in a fixed device array of the library, for
callers that cannot call cudaMalloc (a framework's caching allocator that
owns device memory, a fixed memory budget, a step that must not stall on an
allocation).  Each test calls it through the C ABI and compares it with the
existing two-pass rowwise path of fp8_quantize, byte for byte (the tolerance
of every quantize test here: bytes, scales and amax bit-exact).

The file name makes pytest collect it last; it needs nothing from the other
test files and also passes in a fresh process on its own."""
import numpy as np
import pytest
import torch

import fp8_mixed_precision_scale_gb300 as fp8
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
ROWWISE = fp8.Recipe(kind=fp8.ROWWISE)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    fp8.load_library()


def buffers(rows, cols, layouts):
    """Output buffers of one call, filled with junk so stale bytes show."""
    ld_colT = max(16, (rows + 15) // 16 * 16)
    b = dict(ld_colT=ld_colT, amax=torch.full((1,), 123.0, device=DEV),
             q_row=torch.full((rows, cols), 0x5A, dtype=torch.uint8, device=DEV) if layouts & 1 else None,
             s_row=torch.full((max(rows, 1),), -7.0, device=DEV) if layouts & 1 else None,
             q_colT=torch.full((cols, ld_colT), 0x5A, dtype=torch.uint8, device=DEV) if layouts & 2 else None,
             s_col=torch.full((cols,), -7.0, device=DEV) if layouts & 2 else None)
    return b


def call_no_alloc(x, fmt, layouts, margin=0, stream=None):
    """One call of the no-allocation entry point through the C ABI."""
    rows, cols = x.shape
    b = buffers(rows, cols, layouts)
    rc = fp8.fp8_quantize_rowwise_resident(x, rows, cols, x.stride(0), fmt, margin, layouts, b["amax"], b["q_row"],
                                           b["s_row"], b["q_colT"], b["ld_colT"], b["s_col"], stream, check=False)
    assert rc == 0, fp8.STATUS.get(rc, rc)
    return b


def call_two_pass(x, fmt, layouts, margin=0):
    """The same tensor through fp8_quantize's rowwise path."""
    rows, cols = x.shape
    b = buffers(rows, cols, layouts)
    rc = fp8.fp8_quantize(x, rows, cols, x.stride(0), fmt, fp8.Recipe(kind=fp8.ROWWISE, margin=margin), layouts,
                          None, b["amax"], b["q_row"], b["s_row"], b["q_colT"], b["ld_colT"], b["s_col"], None, 0,
                          check=False)
    assert rc == 0, fp8.STATUS.get(rc, rc)
    return b


def assert_same(got, ref, rows, layouts, what):
    if layouts & 1:
        assert torch.equal(got["q_row"], ref["q_row"]), what + " q_row"
        assert torch.equal(got["s_row"][:rows].view(torch.int32), ref["s_row"][:rows].view(torch.int32)), \
            what + " scale_inv_row"
    if layouts & 2:
        assert torch.equal(got["q_colT"][:, :rows], ref["q_colT"][:, :rows]), what + " q_colT"
        assert torch.equal(got["s_col"].view(torch.int32), ref["s_col"].view(torch.int32)), what + " scale_inv_col"
    assert torch.equal(got["amax"].view(torch.int32), ref["amax"].view(torch.int32)), what + " amax"


def test_two_calls_in_a_row_equal_two_pass_path():
    """The Llama-3-8B activation X [8192, 4096] (Student-t, nu = 4) and a
    ragged [3000, 4104] gradient: two calls in a row of the no-allocation
    entry point, each equal to fp8_quantize's rowwise path."""
    g = torch.Generator().manual_seed(3)
    cases = [(synth.student_t((8192, 4096), 4, g).to(DEV), fp8.E4M3FN),
             ((torch.randn((3000, 4104), generator=g) * 1e-3).to(torch.bfloat16).to(DEV), fp8.E5M2)]
    for x, fmt in cases:
        ref = call_two_pass(x, fmt, 3)
        for i in range(2):
            got = call_no_alloc(x, fmt, 3)
            assert fp8.fp8_sync_status() == 0
            assert_same(got, ref, x.shape[0], 3, f"{tuple(x.shape)} call {i}")


def test_every_counter_reused():
    """70 calls on one stream (the 64 counters of the array are each taken
    more than once): every output equals the two-pass path's, and no barrier
    wait gives up."""
    g = torch.Generator().manual_seed(70)
    xs = [(torch.randn((200, 264), generator=g) * (0.5 + i)).to(torch.bfloat16).to(DEV) for i in range(3)]
    refs = [call_two_pass(x, fp8.E4M3FN, 3, margin=1) for x in xs]
    outs = [call_no_alloc(xs[i % 3], fp8.E4M3FN, 3, margin=1) for i in range(70)]
    assert fp8.fp8_sync_status() == 0
    for i, got in enumerate(outs):
        assert_same(got, refs[i % 3], 200, 3, f"call {i}")


@pytest.mark.parametrize("layouts", [2, 3])
def test_empty_tensor(orc, layouts):
    """rows == 0: column scales of 1 and an amax of 0, as fp8_quantize writes
    them and as the oracle defines them."""
    cols = 136
    x = torch.zeros((0, cols), dtype=torch.bfloat16, device=DEV)
    got = call_no_alloc(x, fp8.E4M3FN, layouts)
    ref = call_two_pass(x, fp8.E4M3FN, layouts)
    assert fp8.fp8_sync_status() == 0
    assert_same(got, ref, 0, layouts, f"empty, layouts {layouts}")
    o = orc.quantize(np.zeros((0, cols), np.uint16), orc.E4M3FN, orc.ROWWISE, layouts=layouts)
    assert np.array_equal(got["s_col"].cpu().numpy().view(np.uint32),
                          np.asarray(o["scale_inv_col"], np.float32).view(np.uint32))
    assert float(got["amax"].cpu()[0]) == float(o["amax"]) == 0.0
