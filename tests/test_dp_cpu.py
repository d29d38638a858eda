"""Data-parallel exchange of the delayed recipe on CPU ranks (gloo, world 2).

Each rank holds a shard of the token rows.  After the ranks' quantize-side
amaxes are MAX-reduced (fp8_mixed_precision_scale_gb300.dp), the oracle's
history update on every rank must equal the single-process update on the
whole tensor -- over several steps, so the rolled history agrees too.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _shards(step, world):
    g = torch.Generator().manual_seed(100 + step)
    full = (torch.randn((64, 48), generator=g) * (1 + step)).to(torch.bfloat16)
    full2 = (torch.randn((64, 24), generator=g) * 1e-3).to(torch.bfloat16)
    return [(full.chunk(world)[r], full2.chunk(world)[r]) for r in range(world)], (full, full2)


def _rank_main(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        import oracle
        import synth
        from fp8_mixed_precision_scale_gb300 import dp
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        L, n = 4, 2
        hist = torch.zeros((n, L), dtype=torch.float32)
        scale = np.ones(n, np.float32)
        sinv = np.ones(n, np.float32)
        fmts = np.array([0, 1], np.uint8)
        for step in range(6):
            shards, _ = _shards(step, world)
            for i, t in enumerate(shards[rank]):
                hist[i, 0] = float(max(hist[i, 0].item(), oracle.amax_bf16(synth.bf16_bits(t))))
            dp.reduce_current_amax(hist)
            h = hist.numpy()
            oracle.update_amax_history(h, scale, sinv, fmts, oracle.MAX, 0)
        q.put((rank, hist.numpy().copy(), scale.copy(), sinv.copy()))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, repr(e), None, None))


def test_amax_allreduce_matches_single_process():
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # single-process reference over the unsharded tensors
    L, n = 4, 2
    hist = np.zeros((n, L), np.float32)
    scale = np.ones(n, np.float32)
    sinv = np.ones(n, np.float32)
    for step in range(6):
        _, full = _shards(step, world)
        for i, t in enumerate(full):
            hist[i, 0] = max(hist[i, 0], oracle.amax_bf16(synth.bf16_bits(t)))
        oracle.update_amax_history(hist, scale, sinv, np.array([0, 1], np.uint8), oracle.MAX, 0)
    for rank, h, s, si in results:
        assert s is not None, h
        assert np.array_equal(h, hist), rank
        assert np.array_equal(s, scale) and np.array_equal(si, sinv), rank


def test_reduce_is_noop_without_process_group():
    from fp8_mixed_precision_scale_gb300 import dp
    h = torch.arange(8, dtype=torch.float32).view(2, 4)
    dp.reduce_current_amax(h)
    assert torch.equal(h, torch.arange(8, dtype=torch.float32).view(2, 4))
