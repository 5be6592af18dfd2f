"""Host logic of the multi-GPU bench path (replicas, one per rank) on CPU
with world_size 2 over gloo: barrier, max-over-ranks timing, whole-job
throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist.barrier()
    ms = [1.0 + rank, 0.5 * (2 - rank)]           # rank 0: [1.0, 1.0]; rank 1: [2.0, 0.5]
    mx = bench.max_over_ranks(ms, dist, "cpu")
    val = bench.job_throughput(w, 1e12, mx[0])
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_rank_max_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, val in res:
        assert mx == [2.0, 1.0]
        # 2 replicas x 1e12 FLOP each in the slowest rank's 2 ms
        assert abs(val - 2 * 1e12 / 2e-3 / 1e12) < 1e-9


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None) == [3.0, 4.0]
    assert bench.job_throughput(1, 6.874e11, 0.55) == pytest.approx(1249.8, rel=1e-3)
