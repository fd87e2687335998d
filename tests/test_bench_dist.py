"""bench.py's multi-process helpers on CPU: two gloo ranks (replicas), max over ranks and the
whole-job throughput, as a torchrun launch would use them."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        # each rank "measured" a different step time; the job is as slow as its slowest rank
        t = bench.max_over_ranks(0.010 + 0.005 * rank, world)
        bench.barrier(world)
        out[rank] = (t, bench.whole_job_throughput(1_000_000, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == pytest.approx(0.015) and res[1][0] == pytest.approx(0.015)
    # two replicas of 1e6 elements in 15 ms: 2e6 / 0.015 / 1e9 Gpixel*ch/s
    assert res[0][1] == pytest.approx(2e6 / 0.015 / 1e9)


def test_single_process_helpers_are_identities():
    import bench

    assert bench.max_over_ranks(0.25, 1) == 0.25
    bench.barrier(1)
    assert bench.whole_job_throughput(5_000_000_000, 1, 1.0) == pytest.approx(5.0)
