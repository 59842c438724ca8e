"""The multi-rank path of the benchmark on CPU: two gloo ranks (spawned
processes) check that the ranks' shards of the global batch are disjoint and
cover it, that the max-over-ranks aggregation gives every rank the slowest
rank's times, and that encoding and attending shard by shard gives what one
rank gives over the global batch (here through the oracle, the same host-side
sharding the GPU ranks use).  The path has no data-path collective (the units
are independent sequences), so the time aggregation is the only exchange."""
import os
import socket
import sys

import numpy as np
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


SHARD = dict(per_rank=2, H=2, T=40, d=64, kb=4, vb=3, G=4)


def _shard_planes(start, n):
    """Oracle encoding and attention of global sequences [start, start + n):
    K, V drawn by global sequence index, q sliced from the global batch's."""
    import oracle
    import tq_synth

    S = SHARD
    w = tq_synth.WORKLOADS["sweep"]
    k, v = tq_synth.host_kv(w, B=n, H=S["H"], d=S["d"], n=S["T"], b_offset=start)
    p = oracle.Planes(n, S["H"], S["d"], S["kb"], S["vb"], 48)
    oracle.encode(p, k, v)
    q_all = tq_synth.host_q(tq_synth.WORKLOADS["decode"], 0, B=2 * S["per_rank"], QH=S["G"] * S["H"], d=S["d"])
    out = oracle.attention(p, np.ascontiguousarray(q_all[start:start + n]), S["T"])
    return [a.copy() for a in p.arrays()], out


def _codec_worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, n = bench.rank_shard(rank, world, SHARD["per_rank"])
        mine = _shard_planes(start, n)
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, start, mine))
        if rank == 0:
            queue.put(sorted(gathered, key=lambda x: x[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_codec_path():
    """Each rank encodes its own sequences and attends over them; the ranks'
    cache bytes, joined in rank order, equal one rank's encoding of the global
    batch byte for byte, and so do the attention outputs (the oracle computes
    each (sequence, q-head) on its own)."""
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_codec_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = queue.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    planes_g, out_g = _shard_planes(0, 2 * SHARD["per_rank"])
    assert [(r, s) for r, s, _ in got] == [(0, 0), (1, SHARD["per_rank"])]
    for i, whole in enumerate(planes_g):
        assert np.array_equal(np.concatenate([m[0][i] for _, _, m in got]), whole)
    assert np.array_equal(np.concatenate([m[1] for _, _, m in got]), out_g)


def test_launcher_command_one_rank_per_gpu():
    cmd = bench.launcher_command(4, ["--steps", "3", "--gpus", "4"])
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-5:] == [os.path.abspath(bench.__file__), "--steps", "3", "--gpus", "4"]


def test_rank_shard_single_and_bad_arguments():
    assert bench.rank_shard(0, 1, 32) == (0, 32)
    assert bench.max_over_ranks([3.0, 1.5], 1) == [3.0, 1.5]
    for bad in ((2, 2, 4), (-1, 2, 4), (0, 0, 4), (0, 2, -1)):
        with pytest.raises(ValueError):
            bench.rank_shard(*bad)
