"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks time
different replicas; both see the slowest rank's time and the whole-job
throughput counts every replica's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [3.5, 7.25][rank]
    slow = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
    q.put((rank, slow, bench.job_throughput(1000, world, slow)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [7.25, 7.25]
    assert res[0][2] == pytest.approx(2 * 1000 / 7.25e-3)


def test_single_rank_is_a_no_op():
    assert bench.max_over_ranks(4.0, 1, None) == 4.0
    assert bench.job_throughput(32768, 1, 1.0) == pytest.approx(3.2768e7)
