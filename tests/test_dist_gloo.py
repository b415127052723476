"""The N>1 host logic of bench.py on CPU with gloo, world size 2: each rank
takes its own replica (no data-path collective), timings reduce by MAX, and
the shard helper partitions units without gaps or overlap."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        elapsed = 10.0 + 5.0 * rank
        worst = bench.reduce_max(elapsed, ws, torch.device("cpu"))
        begin, end = bench.shard_range(37, ws, r)
        q.put((rank, worst, begin, end))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_reduction_and_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2:] == (0, 19) and res[1][2:] == (19, 37)


@pytest.mark.parametrize("total,world", [(32, 1), (32, 2), (7, 4), (3, 8), (64, 8)])
def test_shard_range_partitions(total, world):
    seen = []
    for r in range(world):
        b, e = bench.shard_range(total, world, r)
        assert 0 <= b <= e <= total
        seen.extend(range(b, e))
    assert seen == list(range(total))


def test_batch_split_covers_the_workload():
    """--split batch: the ranks' batch slices of the bench workload are
    disjoint and add up to the one-GPU batch, and so do their KV bytes."""
    from compressed_kv_cache_kvc_gb300 import workloads as W
    w = W.WORKLOADS[bench.WORKLOAD]
    for world in (1, 2, 4, 8):
        slices = [bench.shard_range(w.batch, world, r) for r in range(world)]
        assert slices[0][0] == 0 and slices[-1][1] == w.batch
        assert all(a[1] == b[0] for a, b in zip(slices, slices[1:]))
        per_rank = sum(bench.kv_read_bytes_per_step(w, 100, 3, batch=e - b) for b, e in slices)
        assert per_rank == bench.kv_read_bytes_per_step(w, 100, 3)
