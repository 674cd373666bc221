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


def test_bench_percentiles_and_mask_info_rate():
    import bench
    import workloads
    assert bench.percentiles([5.0, 1.0, 3.0, 2.0, 4.0]) == [1.0, 3.0, 5.0]
    assert bench.percentiles(list(range(1, 101))) == [10, 50, 90]
    w = workloads.workload(2)
    # dense causal, 128 x 128 blocks: 32 x 32 grid, 528 active blocks, 1 pattern
    r = bench.mask_info_rate(w, {"num_active": 528, "num_patterns": 1},
                             {"batch_rows": 1, "nq": 32, "nk": 32}, [0.02, 0.01, 0.03], {"hbm_gbs": 1000.0})
    expect = 32 * 32 + 4 * 33 + 528 * 14 + 128 * 128 // 8
    assert r["bytes"] == expect and r["ms_p50"] == 0.02
    assert abs(r["gbs"] - expect / 0.02e-3 / 1e9) < 1e-2 and abs(r["frac_of_hbm"] - r["gbs"] / 1000.0) < 1e-4


# (batch, query heads, KV heads): GQA groups of 4 and 3, MHA with an odd head
# count, one KV head, and fewer groups than ranks on some shapes
SHARD_SHAPES = [(2, 32, 8), (1, 6, 2), (3, 5, 5), (1, 7, 1), (2, 12, 3), (1, 2, 1)]


def _shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import block_sparse_flash_gb300 as bsf
    L, d = 8, 4
    res = []
    for B, Hq, Hkv in SHARD_SHAPES:
        b0, b1 = bsf.shard_items(B, Hkv, world, rank)
        src = torch.arange(B * Hq * L * d, dtype=torch.float32).view(B, Hq, L, d)
        k = torch.arange(B * Hkv * L * d, dtype=torch.float32).view(B, Hkv, L, d) + 0.5
        seg = torch.arange(B * L, dtype=torch.int32).view(B, L)
        sv = bsf.shard_views(src, k, k, b0, b1, segment_ids=seg)
        # each group reads its own KV head and its batch row's segment IDs
        kv_ok = all(torch.equal(sv["k"][j, 0], k[g // Hkv, g % Hkv]) and torch.equal(sv["segment_ids"][j], seg[g // Hkv])
                    for j, g in enumerate(range(b0, b1)))
        # stand-in for the forward: out = q + 1, lse = q[..., 0], written for this rank's groups only
        pieces = [None] * world
        dist.all_gather_object(pieces, (b0, b1, sv["q"] + 1, sv["q"][..., 0].contiguous()))
        out, lse, cover = bench.gather_shards(pieces, B, Hq, Hkv, L, d)
        res.append((kv_ok, bool((cover == 1).all()), torch.equal(out, src + 1), torch.equal(lse, src[..., 0]),
                    b1 - b0))
    q.put((rank, res))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_split_heads_and_tile_the_output():
    from block_sparse_flash_gb300 import build as b
    b.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for i, (B, Hq, Hkv) in enumerate(SHARD_SHAPES):
        n = [res[r][i][4] for r in range(2)]
        assert sum(n) == B * Hkv and abs(n[0] - n[1]) <= 1, (B, Hq, Hkv, n)
        for r in range(2):
            kv_ok, tiles, out_ok, lse_ok, _ = res[r][i]
            assert kv_ok and tiles and out_ok and lse_ok, (B, Hq, Hkv, r)
