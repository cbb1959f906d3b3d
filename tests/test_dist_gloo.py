"""World-size-2 gloo tests (CPU) of the multi-rank host logic: build agreement, max over ranks and
shard assignment, run as two spawned processes."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from x3x3_convolution_gb300 import dist as xd


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out = {
            "all_ok": xd.agree_all(True),
            "one_failed": xd.agree_all(rank != 1),       # rank 1 could not build: everyone falls back
            "max": xd.max_over_ranks(10.0 + rank),
            "shard": list(xd.shard(7, rank, world)),
        }
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert results[r]["all_ok"] is True
        assert results[r]["one_failed"] is False
        assert results[r]["max"] == 11.0
    assert results[0]["shard"] + results[1]["shard"] == list(range(7))


def test_shard_single_process():
    assert sorted(i for r in range(3) for i in xd.shard(10, r, 3)) == list(range(10))
    assert [len(xd.shard(10, r, 3)) for r in range(3)] == [4, 3, 3]
    with pytest.raises(ValueError):
        xd.shard(5, 2, 2)
    assert xd.agree_all(False) is False and xd.max_over_ranks(3.5) == 3.5
