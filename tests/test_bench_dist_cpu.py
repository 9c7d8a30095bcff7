"""The bench's multi-rank plumbing on CPU: two gloo ranks (one process each, as
torchrun launches them) meet at the barrier, agree on the slowest rank's time, and
the reference arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(2.0 + 3.0 * rank, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((rank, slowest))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], f"rank exit codes {codes}"
    got = dict(out.get(timeout=5) for _ in range(world))
    assert got == {0: 5.0, 1: 5.0}


def test_single_rank_needs_no_process_group():
    bench.dist_init(1, "gloo")
    bench.barrier(1)
    assert bench.max_over_ranks(1.25, 1) == 1.25


@pytest.mark.parametrize("ms,world,expected", [(4.0, 1, 250.0), (4.0, 2, 500.0), (5.0, 8, 1600.0)])
def test_replicas_report_whole_job_throughput(ms, world, expected):
    assert bench.whole_job_steps_per_s(ms, world) == pytest.approx(expected)


def test_reference_arm_does_nothing_off_rank_zero():
    class Args:
        steps, warmup = 3, 3
    # rank 1 of 2 returns before importing torch, building or timing anything
    assert bench.run_reference(Args(), 1, 2, 1) is None
