"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the job
time is the slowest rank's, and throughput aggregates all ranks' tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [100.0, 150.0][rank]
    tot, value = bench.aggregate(local_ms, world, tokens_per_rank=65536, steps=10)
    bench.barrier(world)
    q.put((rank, tot, value))
    dist.destroy_process_group()


def test_aggregate_uses_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tot, value in res:
        assert tot == pytest.approx(150.0)
        assert value == pytest.approx(2 * 65536 * 10 / 0.150)


def test_single_rank_is_identity():
    import bench

    tot, value = bench.aggregate(200.0, 1, tokens_per_rank=1000, steps=4)
    assert tot == 200.0 and value == pytest.approx(4 * 1000 / 0.2)
