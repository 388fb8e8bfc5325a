"""The bench's multi-rank logic on CPU: two gloo ranks, as torchrun would start them.

The step does not shard (replicas only), so the only cross-rank code is the timing: a barrier,
the job time as the largest rank time, and the whole-job throughput over all ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    bench.init_ranks(world, backend="gloo")  # CPU ranks, whatever the machine has
    try:
        assert dist.get_backend() == "gloo"
        bench.barrier(world)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, device="cpu")  # rank 1 is the slow one
        out[rank] = (ms, bench.job_throughput(world, 1000, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_job_time_and_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert set(out.keys()) == {0, 1}
    for rank in range(world):
        ms, steps_per_s = out[rank]
        assert ms == 15.0  # the slowest rank's time, on every rank
        assert steps_per_s == pytest.approx(2 * 1000 / 0.015)  # 2 replicas x 1000 steps in 15 ms


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(1, 500, 250.0) == pytest.approx(2000.0)
