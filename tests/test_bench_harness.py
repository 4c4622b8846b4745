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


def test_reference_arm_json_line_contract():
    """`bench.py --impl reference` as the driver launches it prints exactly
    one JSON line with the contract's keys (run on the tiny workload)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "1",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_rejected():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "2"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_oracle_rate_weights_groups_by_count():
    """A mixed workload's CPU rate weights each wide shape's time per matrix
    by how many matrices of it the workload holds (tall groups count as
    their wide transpose)."""
    import bench
    from newton_schulz_03_gb300.workloads import GroupSpec, Workload
    w = Workload("mixed", "test", (GroupSpec("a", 64, 128, 6), GroupSpec("b", 256, 128, 1),
                                   GroupSpec("c", 128, 256, 2)))
    assert bench.workload_rate(w, {(64, 128): 1.0, (128, 256): 2.0}) == pytest.approx(9 / 12)
    per, done, secs = bench.oracle_shape_seconds(w, 1)
    assert set(per) == {(64, 128), (128, 256)} and done == 2 and secs > 0
