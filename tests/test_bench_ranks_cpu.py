"""The multi-rank (replica) path of bench.py on CPU: two gloo ranks, each with its
own step time, must both see the MAX, and the job throughput counts every
replica's work over that slowest time."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [3.0, 5.0][rank]
    got = bench.max_over_ranks(local, dist, torch.device("cpu"))
    q.put((rank, got, bench.job_throughput(world, 10 ** 12, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
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
    assert [r[1] for r in res] == [5.0, 5.0]
    # 2 replicas x 1 TFLOP in 5 ms -> 400 TFLOP/s
    assert all(abs(r[2] - 400.0) < 1e-9 for r in res)


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert abs(bench.job_throughput(1, 2 * 10 ** 12, 4.0) - 500.0) < 1e-9


def test_cpu_model_is_named():
    import bench
    name = bench.cpu_model()
    assert isinstance(name, str) and name.strip()
