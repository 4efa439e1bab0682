"""Host logic of bench.py that needs no GPU: the max-over-ranks timing reduction of the
replica runs (gloo, world size 2, on CPU) and the ring schedule of the binding."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = bench.max_over_ranks(1.5 + rank, dist)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5


def test_max_over_ranks_without_process_group():
    import bench
    assert bench.max_over_ranks(3.25, None) == 3.25


def test_ring_schedule():
    import context_attention_metadata_gb300 as M
    s = M.ring_schedule(4)
    assert len(s) == 16
    # r-major; at step s shard r meets kv shard (r - s) mod P; first flag on step 0
    assert s[:4] == [(0, 0, True), (0, 3, False), (0, 2, False), (0, 1, False)]
    for r in range(4):
        assert sorted(j for rr, j, _ in s if rr == r) == [0, 1, 2, 3]
    assert M.ring_schedule(4, needed=True) == [(r, M.KV_NEEDED, True) for r in range(4)]
