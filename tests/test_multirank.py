"""The benchmark's multi-rank path on CPU (two gloo ranks): every rank draws
its own batch, the step time is the slowest rank's, and the job's queries/s
counts every rank's batch.  The data path has no collective; the only
exchange is the timing reduction, tested here with the same helpers."""

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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from workloads import Workload, make_inputs
        w = Workload("mr", B=2, Hq=4, Hkv=2, d=64, N=100)
        q, K, V = make_inputs(w, seed=bench.rank_seed(1, rank))
        # each rank's batch is distinct: compare checksums across ranks
        mine = torch.tensor([float(K.float().sum()), float(q.float().sum())], dtype=torch.float64)
        every = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(every, mine)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        value = bench.job_queries_per_s(world, w.B, ms)
        out[rank] = (ms, value, [tuple(t.tolist()) for t in every])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_batches_and_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        ms, value, every = res[r]
        assert ms == 15.0  # the slowest rank's time, on every rank
        assert value == pytest.approx(world * 2 / 15e-3)
        assert every[0] != every[1]  # two different batches
    assert res[0][2] == res[1][2]


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_queries_per_s(1, 16, 0.5) == pytest.approx(32000.0)
    assert len({bench.rank_seed(2, r) for r in range(8)}) == 8
