"""The bench's multi-rank bookkeeping on CPU, two gloo ranks: each rank draws
its own batch, the job time is the slowest rank's, and the job throughput counts
every rank's bytes.  (The data path has no collective: ranks are independent
replicas.)"""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_cache_43_gb300 import workloads as W
        seed = bench.rank_seed(2, rank)
        q_lens, ctx, _ = W.lengths(2, small=True, seed=seed)
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(1e9, world, job_ms)
        q.put((rank, seed, tuple(int(x) for x in ctx), job_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, c0, t0, v0), (r1, s1, c1, t1, v1) = res
    assert s0 != s1 and c0 != c1                  # independent batches
    assert t0 == t1 == 15.0                        # slowest rank's time on both
    assert v0 == v1 == pytest.approx(2 * 1e9 / 15e-3 / 1e9)
