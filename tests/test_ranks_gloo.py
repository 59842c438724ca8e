"""The multi-rank path of the benchmark on CPU: two gloo ranks (spawned
processes) check that the ranks' shards of the global batch are disjoint and
cover it, and that the max-over-ranks aggregation gives every rank the
slowest rank's times.  The path has no data-path collective (the units are
independent sequences), so this aggregation is the only exchange."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, n = bench.rank_shard(rank, world, 4)
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.0 * rank], world, "cpu")
        queue.put((rank, start, n, times))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_aggregate():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, s, n) for r, s, n, _ in got] == [(0, 0, 4), (1, 4, 4)]  # disjoint, covering [0, 8)
    for _, _, _, times in got:
        assert times == [2.0, 5.0, 2.0]


def test_rank_shard_single_and_bad_arguments():
    assert bench.rank_shard(0, 1, 32) == (0, 32)
    assert bench.max_over_ranks([3.0, 1.5], 1) == [3.0, 1.5]
    for bad in ((2, 2, 4), (-1, 2, 4), (0, 0, 4), (0, 2, -1)):
        with pytest.raises(ValueError):
            bench.rank_shard(*bad)
