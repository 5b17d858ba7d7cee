"""The multi-GPU mode of bench.py: N independent replicas (no data-path
collective), each rank with its own seeded batch, the step time taken as the max
over ranks and the throughput as the whole-job aggregate.  The rank logic runs
here as two gloo processes on the CPU."""
import dataclasses
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # each replica's timing differs; every rank must see the same maximum
        ms = 10.0 + 5.0 * rank
        mx = bench.reduce_max(ms, w)
        seed = bench.rank_seed(W.workload("tiny").seed, r)
        x = W.make_x(dataclasses.replace(W.workload("tiny"), seed=seed))
        out[rank] = (mx, seed, float(x.float().sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_distinct_batches():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0           # max over ranks, identical everywhere
    assert res[0][1] != res[1][1]                   # distinct seeds per rank
    assert res[0][2] != res[1][2]                   # hence distinct batches


def test_throughput_is_whole_job_aggregate():
    # 2 ranks x 16384 tokens x 10 steps in 20 ms (max over ranks) -> 16.384 M tokens/s
    assert bench.throughput(16384, 2, 10, 20.0) == pytest.approx(16384 * 2 * 10 / 0.020)
    assert bench.throughput(16384, 1, 10, 20.0) * 2 == pytest.approx(bench.throughput(16384, 2, 10, 20.0))


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.rank_seed(1000, 0) == 1000
