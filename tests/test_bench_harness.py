"""The benchmark's multi-rank harness on CPU (gloo, world size 2): barrier,
max-over-ranks timing, the job value over the slowest rank, the ranks' shares
of the workload, the end-to-end host passes and the CPU baseline's sample."""

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


def test_job_value_over_the_slowest_rank():
    """The ranks share one workload: the job value is the workload's
    matrices per step over the slowest rank's time, whatever the rank count."""
    import bench
    assert bench.job_value(1030, 20, 10.0) == pytest.approx(2060.0)
    assert bench.job_value(1030, 20, 5.0) == pytest.approx(2 * bench.job_value(1030, 20, 10.0))


def test_e2e_host_passes_fit_the_budget():
    """The end-to-end leg holds 1/P of every group whose count P divides:
    the L=102 layer (226 GB of FP32 state) needs P = 4 under a 98 GB host
    budget (58 GB held) and P = 64 under the leg's 12 GiB pinned budget
    (3.4 GB of experts + the 6.3 GB shared expert and attention held
    whole); a workload that fits is held whole."""
    import bench
    from newton_schulz_03_gb300.workloads import WORKLOADS
    w = WORKLOADS["l102_layer"]
    counts = [g.count for g in w.groups]
    elems = [g.rows * g.cols for g in w.groups]
    assert bench.e2e_passes(counts, elems, 98 << 30) == 4
    assert bench.e2e_passes(counts, elems, bench.E2E_HOST_BYTES) == 64
    assert bench.e2e_passes(counts, elems, 300 << 30) == 1
    w24 = WORKLOADS["l24_attention"]
    assert bench.e2e_passes([96], [2048 * 2048], 98 << 30) == 1
    assert bench.e2e_passes([w24.groups[0].count], [2048 * 2048], 1 << 30) == 8


def test_rank_shares_partition_the_workload():
    """bench.py's ranks step disjoint slices that cover the workload."""
    import bench
    from newton_schulz_03_gb300.workloads import WORKLOADS
    w = WORKLOADS["l102_layer"]
    for world in (1, 2, 4, 8):
        seen = {}
        for rank in range(world):
            for gi, first, count in bench.rank_share(w, world, rank):
                seen.setdefault(gi, []).append((first, count))
        for gi, g in enumerate(w.groups):
            spans = sorted(seen[gi])
            assert spans[0][0] == 0 and sum(c for _, c in spans) == g.count
            assert all(a + c == b for (a, c), (b, _) in zip(spans, spans[1:]))


def test_cpu_baseline_extrapolates_shapes_too_long_for_the_sample():
    """On the L=102 layer the oracle times the 2048 x 8704 experts and
    extrapolates 8704 x 8704 and 8704 x 13056 (tens of seconds each) by
    their flop count at the measured FP64 rate."""
    import bench
    from newton_schulz_03_gb300.workloads import WORKLOADS
    w = WORKLOADS["l102_layer"]
    per = {(2048, 8704): 2.0}
    full = bench.complete_per_matrix(w, per, [(8704, 8704), (8704, 13056)])
    f = bench.oracle_flops
    assert full[(8704, 8704)] == pytest.approx(2.0 * f(8704, 8704, 5) / f(2048, 8704, 5))
    assert full[(8704, 13056)] == pytest.approx(2.0 * f(8704, 13056, 5) / f(2048, 8704, 5))
    text = bench.oracle_sample_text(w, 3, "", [(2048, 8704)], [(8704, 8704), (8704, 13056)])
    assert "extrapolated" in text and "8704x13056" in text


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


def test_default_step_count():
    """About 5 s of steps: 10 to 100, or 3 when one step takes over 0.6 s."""
    import bench
    assert bench.step_count(7e-5) == 100          # tiny
    assert bench.step_count(0.012) == 100         # l24
    assert bench.step_count(0.133) == 38          # l48 experts
    assert bench.step_count(0.49) == 11           # L=102 layer
    assert bench.step_count(0.6) == 10
    assert bench.step_count(6.7) == 3             # 48-layer model


def test_energy_of_a_step():
    import bench
    e = bench.energy_of_step({"power_w_median": 1400.0}, 500.0, 7.0e14)
    assert e["joules_per_step"] == 700.0
    assert e["tflop_per_joule"] == pytest.approx(1.0)
    assert bench.energy_of_step({"sm_mhz": None}, 500.0, 7.0e14) is None
