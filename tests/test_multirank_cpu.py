"""The multi-rank (replica) host logic of bench.py with 2 gloo ranks on CPU."""

import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_fp8_kv_cache_gb300 import workloads


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local = [10.0 + rank, 3.0 * (world - rank)]  # per-rank timings (ms)
        got = bench.max_over_ranks(local, dist, "cpu")
        spec = workloads.CONFIGS[2]
        q.put((rank, got, bench.rank_seed(spec, rank)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_timings():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [[11.0, 6.0], [11.0, 6.0]]
    seeds = [r[2] for r in res]
    assert seeds[0] == workloads.CONFIGS[2].seed and len(set(seeds)) == 2  # distinct batches per rank


def test_aggregate_is_weak_scaling_total():
    # 2 ranks x 5 steps x 1e9 bytes in 10 ms (slowest rank) -> 1000 GB/s
    assert bench.aggregate_gbs(10 ** 9, 2, 5, 10.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]  # single process: unchanged
