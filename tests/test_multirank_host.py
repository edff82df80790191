"""The N > 1 path of bench.py, on the CPU: two gloo ranks (one process each,
as torchrun starts them) check that every rank draws its own batch, that the
job's times are the slowest rank's, that the whole-job rate counts the work of
all ranks, and that only rank 0 runs the reference arm and prints."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    from causal_head_self_gb300 import inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = inputs.WORKLOADS[bench.PREFILL]
        # each rank's own batch: a small slice of its inputs, compared across ranks
        q, _, _ = inputs.prefill_inputs(1, 1, 1, 8, 64, bench.rank_seed(w["seed"], rank))
        mine = q.float().flatten()
        got = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        distinct = not torch.equal(got[0], got[1])
        # rank r took (1 + r) and (10 - r) seconds: the job's times are the maxima
        t = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world)
        rate = bench.job_rate(100.0, t[0], world)

        class A:
            steps, warmup, gpus = 1, 3, world
        ref = bench.run_reference(A(), rank, world) if rank != 0 else "rank 0 runs it"
        results[rank] = (distinct, t, rate, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    for rank in range(world):
        distinct, t, rate, ref = res[rank]
        assert distinct
        assert t == [2.0, 10.0]
        assert rate == pytest.approx(100.0 * world / 2.0)
    assert res[1][3] is None   # non-zero ranks leave the reference arm without work


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_rate(50.0, 2.0, 1) == 25.0
    assert bench.rank_seed(7, 0) == 7 and bench.rank_seed(7, 1) != 7
