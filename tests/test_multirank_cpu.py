"""The bench's multi-rank bookkeeping on CPU: two gloo ranks (world size 2) each time
their own replica of the workload; the job reports the slowest rank's time and the
work of both ranks.  No GPU and no data-path collective are involved: the path shards
into independent replicas."""
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


def _rank_main(rank, world, port, results):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [0.25, 0.40][rank]  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(torch, dist, mine, torch.device("cpu"))
        dist.barrier()
        results[rank] = (slowest, bench.whole_job_rate(world, 1e12, 10, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_all_work():
    port = _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, rate = results[r]
        assert slowest == pytest.approx(0.40)
        assert rate == pytest.approx(2 * 1e12 * 10 / 0.40 / 1e12)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, None, 1.5, torch.device("cpu")) == 1.5
    assert bench.whole_job_rate(1, 2e12, 4, 2.0) == pytest.approx(4.0)
