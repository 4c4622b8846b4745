"""The benchmark's own arm on the GPU: one JSON line with the contract's
keys (tiny workload, end-to-end leg and CPU baseline included)."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line_contract():
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "1", "--workload", "tiny",
                        "--steps", "5", "--warmup", "3", "--cpu-seconds", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["steps"] == 5 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny" and d["scaling"] == "strong"
    # 18 library launches per step (cast, norm, 5 x 3 products, apply)
    assert d["gpu_launches"] == 18 * 5
    rf = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] == "tensor" and rf["achieved"] > 0 and rf["frac"] > 0
    # frac is against the measured burst peak; the sustained one is beside it
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    assert rf["frac_of_sustained"] == pytest.approx(rf["achieved"] / rf["peak_sustained"],
                                                    rel=1e-3)
    assert rf["achieved"] == pytest.approx(rf["flops_per_launch"] / (rf["avg_launch_ms"] * 1e9),
                                           rel=1e-4)
    # Every kernel's average launch time from the same event pass.
    assert rf["kernel_avg_launch_ms"]["ns_update"] == pytest.approx(rf["avg_launch_ms"], rel=1e-4)
    assert set(rf["kernel_avg_launch_ms"]) >= {"momentum_cast", "ns_gram", "ns_poly", "ns_update",
                                                "apply"}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    # tiny: 4 matrices of 128 x 64, M, G, W in (12 B/element), M, W out (8 B)
    assert e["h2d_bytes_per_step"] == 4 * 128 * 64 * 12
    assert e["d2h_bytes_per_step"] == 4 * 128 * 64 * 8
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    en = d["energy"]
    if en is not None:      # None only when nvidia-smi gave no samples
        assert en["joules_per_step"] == pytest.approx(
            en["power_w_median"] * d["ms_per_step"] / 1e3, rel=1e-3)
    # Steps under 1 ms are timed as a block only (no per-step events).
    assert d["ms_per_step_median"] is None and d["ms_per_step_min_max"] is None


def test_bench_reports_the_median_step():
    """Steps of 1 ms or more: an event after every step gives the median
    and the extremes of the K step times beside the block time."""
    r = subprocess.run([sys.executable, "bench.py", "--workload", "l24_attention",
                        "--max-count", "16", "--steps", "10", "--warmup", "3", "--skip-e2e",
                        "--skip-cpu-baseline"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1])
    lo, hi = d["ms_per_step_min_max"]
    assert 0 < lo <= d["ms_per_step_median"] <= hi
    # The block time per step is the mean of the same K steps.
    assert lo * 0.999 <= d["ms_per_step"] <= hi * 1.001
