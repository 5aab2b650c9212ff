"""The benchmark's multi-GPU arm runs independent replicas (the decode path
shards by sequence with no exchange) and reports the slowest rank's time.
Here two gloo ranks on the CPU exercise that host-side logic: the barrier
and the max-over-ranks reduction of the timed region, and the whole-job
throughput built from it."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._env_rank() == (rank, world, rank)
        bench._barrier(world)
        local_time = 0.25 + 0.5 * rank           # rank 1 is the slow one
        t_max = bench._max_over_ranks(local_time, world)
        bytes_per_rank = 1000.0
        results[rank] = (t_max, world * bytes_per_rank / t_max)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_report_slowest_rank():
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 0.75
    assert results[0][1] == pytest.approx(2000.0 / 0.75)


def test_single_rank_passthrough():
    import bench
    assert bench._max_over_ranks(1.5, 1) == 1.5
    bench._barrier(1)
