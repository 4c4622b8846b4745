"""The benchmark's multi-rank harness on CPU (gloo, world size 2): barrier,
max-over-ranks timing and the weak-scaling job value."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr_ = bench.dist_env()
    assert (w, r, lr_) == (world, rank, rank)
    bench.barrier(world)
    # Rank r pretends its timed region took 1 + r seconds.
    slowest = bench.max_over_ranks(1.0 + rank, world)
    out[rank] = slowest
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_job_value_weak_scaling():
    import bench
    one = bench.job_value(1, 96, 20, 0.3)
    two = bench.job_value(2, 96, 20, 0.3)
    assert two == pytest.approx(2 * one)
    assert bench.job_value(4, 96, 20, 0.6) == pytest.approx(2 * one)


def test_reference_arm_other_ranks_exit_quietly():
    import argparse
    import bench
    args = argparse.Namespace(workload="tiny", steps=1, warmup=3)
    assert bench.run_reference(args, world=2, rank=1) is None
    line = bench.run_reference(args, world=1, rank=0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
