"""The N>1 bench path on CPU: two gloo ranks, each with its own per-step time,
must agree on the max over ranks and on the whole-job throughput (every rank
processes its own copy of the workload: weak scaling, no data-path collective)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 + rank  # rank 1 is the slowest
    m = bench.reduce_max(ms, world, device=torch.device("cpu"))
    value = bench.whole_job_throughput(1e12, world, m)
    q.put((rank, m, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
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
    for rank, m, value in res:
        assert m == pytest.approx(3.0)
        assert value == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(1.5, 1) == 1.5
    assert bench.whole_job_throughput(2e12, 1, 2.0) == pytest.approx(1000.0)
