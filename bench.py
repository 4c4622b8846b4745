"""Benchmark of the one-GPU Muon step: NS-orthogonalised matrices/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one muon_step over the workload's parameter groups: momentum
update + BF16 cast, Newton-Schulz on every matrix, weight update.  The
default workload is one full-scale layer of the largest model (L=102,
hidden 8704: 1024 expert matrices of 2048 x 8704, the shared expert and
four 8704 x 8704 attention projections; 226 GB of FP32 state).  Inputs are
seeded synthetic tensors resident in HBM and larger than L2, so no flush is
needed between steps.  With N > 1 (torchrun) the workload's whole matrices
are split over the ranks by muon_partition (longest processing time
first); every rank steps its own share with no exchange, and the job value
is the workload's matrices over the slowest rank's time.

The JSON line adds the roofline of the dominant kernel (the Newton-Schulz
update product), measured live with CUDA events on the launching stream,
the CPU oracle timed on a bounded sample (rank 0, N = 1), and an
end-to-end figure through the host-buffer entry point with the copies
inside the timed region.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NS-orthogonalised matrices/s and TFLOPS (% of GB300 BF16 peak); muon_step ms"
UNIT = "matrices/s"
DEFAULT_WORKLOAD = "l102_layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DOMINANT = "ns_update"
NS_SOURCES = ("newton_schulz_03_gb300/csrc/k_ns_gemm.cu", "newton_schulz_03_gb300/csrc/k_ns_gemm2.cu",
              "newton_schulz_03_gb300/csrc/ns_common.cuh", "newton_schulz_03_gb300/csrc/sm103_ptx.cuh")


# ----------------------------------------------------------------- harness
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sig(x, digits: int = 6):
    """`x` rounded to `digits` significant digits (None stays None)."""
    if x is None:
        return None
    return float(f"{x:.{digits}g}")


def job_value(units_per_step: float, steps: int, secs: float) -> float:
    """Whole-job throughput: the ranks share one workload of
    `units_per_step` matrices per step; the job takes as long as the
    slowest rank."""
    return units_per_step * steps / secs


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def timed_steps(step, steps: int, warmup: int, world: int, stream, sync, per_step=None) -> float:
    """W untimed steps, then K steps between barrier+sync on both sides,
    timed with CUDA events on `stream`.  Returns seconds (max over ranks).
    With a list `per_step`, an event is also recorded after every step and
    the K step durations (ms, this rank) are appended to it; the total is
    still the first event to the last."""
    import torch
    for _ in range(warmup):
        step()
    sync()
    barrier(world)
    sync()
    ev = [torch.cuda.Event(enable_timing=True)
          for _ in range(steps + 1 if per_step is not None else 2)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        if per_step is not None:
            ev[i + 1].record(stream)
    ev[-1].record(stream)
    sync()
    barrier(world)
    secs = ev[0].elapsed_time(ev[-1]) / 1e3
    if per_step is not None:
        per_step.extend(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    return max_over_ranks(secs, world, device=torch.device("cuda", torch.cuda.current_device()))


def step_count(t1: float) -> int:
    """Default K from one step's time: about 5 s of steps (enough clock
    samples), at least 10 steps (3 when a step takes over 0.6 s), at most
    100."""
    k = math.ceil(5.0 / max(t1, 1e-6))
    return int(max(10 if t1 <= 0.6 else 3, min(100, k)))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"muon_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "power_w_max": max(r[2] for r in rows),
                "power_w_median": statistics.median(r[2] for r in loaded),
                "samples": len(loaded), "reasons": reasons}


def energy_of_step(clocks: dict, ms_per_step: float, flops_step: float):
    """Energy per step from the board power sampled during the timed passes
    (median of the samples under load): the products run at the power cap,
    so flops per joule is what bounds their throughput there."""
    w = clocks.get("power_w_median")
    if not w or ms_per_step <= 0:
        return None
    joules = w * ms_per_step / 1e3
    return {"power_w_median": round(w, 1), "joules_per_step": sig(joules),
            "tflop_per_joule": sig(flops_step / 1e12 / joules) if joules > 0 else None,
            "source": "nvidia-smi power.draw every 200 ms during the timed passes"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def ns_source_hash() -> str:
    """Hash of the Newton-Schulz kernel sources with comments and blank
    lines removed: a profile stays valid across comment-only edits."""
    import re
    h = hashlib.sha256()
    for p in NS_SOURCES:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, matrices_per_step: dict, launches_per_step: float):
    """Average DRAM bytes per launch of the dominant kernel from the
    committed ncu summary, if it was taken on the current kernel source.
    The summary gives DRAM bytes per matrix for each wide shape
    (``dram_bytes_per_matrix[MxN]``; traffic grows with the matrix count),
    measured on a small case; one step's launches cover
    ``matrices_per_step[(m, n)]`` matrices of each shape."""
    path = os.path.join(ROOT, "profiles", f"{DOMINANT}_{workload.split('[')[0]}.txt")
    if not os.path.exists(path) or launches_per_step <= 0:
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != ns_source_hash():
        return None
    total = 0.0
    for (m, n), count in matrices_per_step.items():
        key = f"dram_bytes_per_matrix[{m}x{n}]"
        if key not in kv and len(matrices_per_step) == 1:
            key = "dram_bytes_per_matrix"
        try:
            total += float(kv[key]) * count
        except (KeyError, ValueError):
            return None
    return round(total / launches_per_step)


# ----------------------------------------------------------------- our arm
def capped(w, max_count, shape=None):
    """The workload with every group's count capped and, with `shape`
    ("MxN"), only the groups of that wide shape (small profiling cases)."""
    if not max_count and not shape:
        return w
    import dataclasses
    gs = w.groups
    name = w.name
    if shape:
        m, n = (int(v) for v in shape.lower().split("x"))
        gs = tuple(g for g in gs if g.wide == (m, n))
        if not gs:
            raise SystemExit(f"workload {w.name} has no group of wide shape {shape}")
        name += f"[{m}x{n}]"
    if max_count:
        gs = tuple(dataclasses.replace(g, count=min(g.count, max_count)) for g in gs)
        name += f"[count<={max_count}]"
    return dataclasses.replace(w, name=name, groups=gs)


def workload_groups(w):
    return [(g.rows, g.cols, g.count) for g in w.groups]


def rank_share(w, world, rank):
    """This rank's slices of the workload: [(group index, first, count)]
    from the library's whole-matrix partition (all of it at world = 1)."""
    import newton_schulz_03_gb300 as ns
    if world == 1:
        return [(gi, 0, g.count) for gi, g in enumerate(w.groups) if g.count > 0]
    slices, _ = ns.muon_partition(workload_groups(w), world, w.ns_steps)
    return slices[rank]


def share_wide_counts(w, share):
    out = {}
    for gi, _, count in share:
        key = w.groups[gi].wide
        out[key] = out.get(key, 0) + count
    return out


def run_ours(args, world, rank, local):
    import torch

    import newton_schulz_03_gb300 as ns
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_torch

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w = capped(WORKLOADS[args.workload], args.max_count, args.shape)
    share = rank_share(w, world, rank)
    groups = [(w.groups[gi].rows, w.groups[gi].cols, count) for gi, _, count in share]
    tensors = [make_group_torch(w, gi, dev, first, count) for gi, first, count in share]
    Ws = [t[0] for t in tensors]
    Ms = [t[1] for t in tensors]
    Gs = [t[2] for t in tensors]
    del tensors
    stream = torch.cuda.current_stream()
    handle = ns.Handle(device=local)
    h = handle.value
    plan_all = ns.muon_plan_describe(workload_groups(w), w.ns_steps)
    layers = w.layers

    def step_on(s):
        # One step of this rank's share: `layers` calls over the resident layer.
        for _ in range(layers):
            ns.muon_step(h, groups, Ms, Gs, Ws, w.lr, w.wd, w.mu, w.ns_steps, s)

    def step():
        step_on(stream)

    sync = torch.cuda.synchronize
    step()
    ns.muon_last_device_error(h, stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    step()
    b.record(stream)
    sync()
    t1 = max_over_ranks(a.elapsed_time(b) / 1e3, world, device=torch.device(dev))
    if args.steps is None:
        args.steps = step_count(t1)
    # Per-step events break launch chaining at one kernel boundary per
    # step: a few microseconds, nothing against steps of 1 ms or more.
    per_step = [] if t1 >= 1e-3 else None
    ns.muon_reset_kernel_stats(h)
    graph_ms = None
    if args.graph:
        # The same step captured once in a CUDA graph and replayed.
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            step_on(cap)
        stream.wait_stream(cap)
        gsecs = timed_steps(g.replay, args.steps, args.warmup, world, stream, sync)
        graph_ms = gsecs * 1e3 / args.steps
        ns.muon_reset_kernel_stats(h)

    with ClockSampler(local) as clk:
        # The step as a user runs it: no per-kernel events.
        ns.muon_reset_kernel_stats(h)
        launches0 = ns.muon_kernel_stats(h)["total_launches"]
        secs = timed_steps(step, args.steps, args.warmup, world, stream, sync, per_step)
        launches1 = ns.muon_kernel_stats(h)["total_launches"]
        # The same K steps again with an event pair around every launch on
        # the launching stream: per-kernel durations for the roofline.  The
        # events serialise the launches, so this pass is a little slower.
        ns.muon_set_kernel_timing(h, True)
        ns.muon_reset_kernel_stats(h)
        secs_ev = timed_steps(step, args.steps, args.warmup, world, stream, sync)
        stats = ns.muon_kernel_stats(h)
        ns.muon_set_kernel_timing(h, False)
    ns.muon_last_device_error(h, stream)
    clocks = clk.summary()
    # Launch and time counts include the warm-up steps; scale to the timed K.
    frac_timed = args.steps / float(args.steps + args.warmup)
    gpu_launches = int(round((launches1 - launches0) * frac_timed))

    matrices_per_step = w.matrices
    value = job_value(matrices_per_step, args.steps, secs)
    ms_per_step = secs * 1e3 / args.steps
    flops_step = plan_all["ns_algorithmic_flops"] * layers
    tflops = flops_step * args.steps / secs / 1e12

    peaks, peak_src = load_peaks()
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    # This rank's kernels: its own share of the workload.
    mine = share_wide_counts(w, share)
    my_flops_step = sum(c * w.ns_steps * (3.0 * m * m * n + m ** 3) for (m, n), c in mine.items()) \
        * layers
    # Dominant kernel: the update product X' = alpha B' X, 2 m^2 n flops per matrix.
    upd_flops_step = sum(c * 2.0 * m * m * n for (m, n), c in mine.items()) * w.ns_steps * layers
    upd_launches = stats["launches"][DOMINANT]
    upd_ms = stats["total_ms"][DOMINANT]
    steps_recorded = args.steps + args.warmup
    achieved = (upd_flops_step * steps_recorded) / (upd_ms / 1e3) / 1e12 if upd_ms > 0 else None
    ns_ms = sum(stats["total_ms"][k] for k in ("ns_gram", "ns_poly", "ns_update"))
    ns_tflops = (my_flops_step * steps_recorded) / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else None
    kernel_share = {k: round(v / max(sum(stats["total_ms"].values()), 1e-9), 4)
                    for k, v in stats["total_ms"].items() if v > 0}
    upd_matrices_step = {k: c * w.ns_steps * layers for k, c in mine.items()}
    traffic = profiled_traffic(w.name, upd_matrices_step, upd_launches / steps_recorded) \
        if upd_launches else None
    roofline = {
        "kernel": ("ns_gemm_pair_kernel<update>" if min(m for m, _ in mine) > 128
                   else "ns_gemm_kernel<update,256>") + " (X' = alpha B' X)",
        "bound": "tensor", "achieved": sig(achieved),
        "peak": burst, "unit": "TFLOP/s",
        "frac": sig(achieved / burst) if achieved else None,
        "peak_source": f"{peak_src} bf16_tflops, burst (of {peak_src})",
        "peak_sustained": sustained,
        "frac_of_sustained": sig(achieved / sustained) if achieved else None,
        "traffic": traffic,
        "traffic_source": (f"profiles/{DOMINANT}_{w.name.split('[')[0]}.txt: ncu DRAM bytes per "
                           "matrix on a small case x matrices per launch" if traffic else None),
        "launches": upd_launches,
        "avg_launch_ms": sig(upd_ms / upd_launches) if upd_launches else None,
        "flops_per_launch": round(upd_flops_step * steps_recorded / upd_launches)
        if upd_launches else None,
        "ns_engine_tflops": sig(ns_tflops),
        "ns_engine_frac": sig(ns_tflops / burst) if ns_tflops else None,
        "ns_engine_frac_of_sustained": sig(ns_tflops / sustained) if ns_tflops else None,
        "kernel_time_share": kernel_share,
        "kernel_avg_launch_ms": {k: sig(stats["total_ms"][k] / n)
                                 for k, n in stats["launches"].items() if n > 0},
    }
    # The HBM-bound kernels against the measured copy bandwidth: 14 B per
    # element for the momentum update + cast (read M, G; write M, X) and
    # 10 B for the apply (read W, O; write W).
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    elems_step = sum(w.groups[gi].rows * w.groups[gi].cols * c for gi, _, c in share) * layers
    hbm_kernels = {}
    for kind, bpe in (("momentum_cast", 14), ("apply", 10)):
        ms = stats["total_ms"].get(kind, 0.0)
        if ms > 0:
            gbs = elems_step * bpe * steps_recorded / (ms / 1e3) / 1e9
            hbm_kernels[kind] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                                 "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                                 "bytes_per_element": bpe}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch RNG on device, shapes of the workload)",
        "config": {
            "workload": w.name, "description": w.description,
            "matrices_per_step": matrices_per_step, "groups": workload_groups(w),
            "layers": layers, "ns_steps": w.ns_steps, "mu": w.mu, "lr": w.lr, "wd": w.wd,
            "precision": "FP32 momentum and weights, BF16 Newton-Schulz with FP32 accumulation",
            "l2": "inputs larger than L2 (%.1f GB of FP32 state per layer), no flush"
                  % (sum(g.numel for g in w.groups) * 12 / 1e9),
            "parallelism": (f"{world} ranks, whole matrices split by muon_partition (LPT), "
                            "no exchange" if world > 1 else "single GPU"),
        },
        "tflops_algorithmic": round(tflops, 1),
        "pct_of_bf16_peak": round(100 * tflops / burst, 2),
        "pct_of_bf16_sustained": round(100 * tflops / sustained, 2),
        "tflops_dense_equivalent": round(tflops * dense_over_alg(w), 1),
        "gpu_launches": gpu_launches,
        "graph_replay_ms_per_step": round(graph_ms, 4) if graph_ms is not None else None,
        "ms_per_step_with_kernel_events": round(secs_ev * 1e3 / args.steps, 4),
        "ms_per_step_median": round(statistics.median(per_step), 4) if per_step else None,
        "ms_per_step_min_max": [round(min(per_step), 4), round(max(per_step), 4)]
        if per_step else None,
        "programmatic_dependent_launch": os.environ.get("MUON_PDL", "1") != "0",
        "clocks": clocks,
        "energy": energy_of_step(clocks, ms_per_step, flops_step),
        "roofline": roofline,
        "hbm_kernels": hbm_kernels,
    }
    if not args.skip_e2e:
        line["e2e"] = run_e2e(args, ns, h, w, share, Ws, Ms, Gs, world)
    if args.adamw:
        line["adamw"] = run_adamw(ns, h, peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        del Ws, Ms, Gs
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    handle.close()
    return line


def run_adamw(ns, h, hbm_peak):
    """The AdamW companion on the non-Muon parameters of a rung-L=24 model
    (untied input and output embeddings of 131072 x 2048, 49 norm vectors of
    2048): 28 bytes per element (read p, g, m, v; write p, m, v)."""
    import torch
    sizes = [131072 * 2048, 131072 * 2048] + [2048] * 49
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    P = [torch.randn(n, generator=gen, device="cuda") for n in sizes]
    G = [torch.randn(n, generator=gen, device="cuda").mul_(1e-3) for n in sizes]
    M = [torch.zeros(n, device="cuda") for n in sizes]
    V = [torch.zeros(n, device="cuda") for n in sizes]
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)
    for t in range(1, 4):
        ns.muon_adamw_step(h, P, G, M, V, step=t, **hp)
    ns.muon_reset_kernel_stats(h)
    ns.muon_set_kernel_timing(h, True)
    steps = 10
    for t in range(4, 4 + steps):
        ns.muon_adamw_step(h, P, G, M, V, step=t, **hp)
    st = ns.muon_kernel_stats(h)
    ns.muon_set_kernel_timing(h, False)
    ns.muon_last_device_error(h)
    n = sum(sizes)
    ms = st["total_ms"]["adamw"] / steps
    gbs = 28.0 * n / (ms / 1e3) / 1e9
    return {"params": n, "ms_per_step": round(ms, 4), "achieved": round(gbs, 1), "unit": "GB/s",
            "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4), "bound": "hbm",
            "bytes_per_element": 28, "launches_per_step": st["launches"]["adamw"] / steps,
            "workload": "rung L=24 non-Muon parameters: 2 x 131072x2048 embeddings + 49 x 2048 norms"}


def dense_over_alg(w) -> float:
    alg = dense = 0.0
    for (m, n), c in w.wide_batches().items():
        alg += c * (3.0 * m * m * n + m ** 3)
        dense += c * (4.0 * m * m * n + 2.0 * m ** 3)
    return dense / alg


def host_available_bytes() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def e2e_passes(group_counts, elems_per_matrix, budget_bytes) -> int:
    """Smallest power of two P such that host buffers holding 1/P of every
    group whose count P divides (and the other groups whole) fit the budget
    (12 bytes per element: momentum, gradient, weights)."""
    p = 1
    while True:
        held = sum((c // p if c % p == 0 else c) * e * 12
                   for c, e in zip(group_counts, elems_per_matrix))
        if held <= budget_bytes or p >= max(group_counts + [1]):
            return p
        p *= 2


# Pinned host footprint of the end-to-end leg.  On the GB300 hosts measured
# here, copies from cudaHostAlloc memory ran at the link's ~200 GB/s each
# way up to 16 GiB of it, and beyond 16-32 GiB (depending on the host) one
# direction fell to 56-100 GB/s; 12 GiB keeps the leg at the link's rate.
E2E_HOST_BYTES = 12 << 30


def run_e2e(args, ns, h, w, share, Ws, Ms, Gs, world):
    """The same step through muon_step_host: page-locked host buffers
    (muon_host_alloc), H2D of momentum, gradient and weights and D2H of
    momentum and weights inside the timed region.

    When the rank's whole share does not fit the pinned host budget (the
    L=102 layer is 226 GB of FP32 state), the host buffers hold 1/P of
    every group whose count P divides (the routed experts) and the others
    whole, and one step is P calls: the first over every group, the other
    P-1 over the divided groups again.  Each step then copies and steps as
    many matrices of each shape as the device step (the same bytes and
    flops); the values of the divided groups repeat."""
    import torch
    counts = [c for _, _, c in share]
    elems = [w.groups[gi].rows * w.groups[gi].cols for gi, _, _ in share]
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_available_bytes() // (2 * max(1, local_ranks))
    budget = min(E2E_HOST_BYTES, avail) if avail > 0 else E2E_HOST_BYTES
    P = e2e_passes(counts, elems, budget)
    held = [c // P if (P > 1 and c % P == 0) else c for c in counts]
    divided = [P > 1 and c % P == 0 for c in counts]
    host = []
    for i, (gi, _, _) in enumerate(share):
        g = w.groups[gi]
        trip = []
        for dev_t in (Ws[i], Ms[i], Gs[i]):
            t = ns.host_empty((held[i], g.rows, g.cols))
            t.copy_(dev_t[:held[i]])
            trip.append(t)
        host.append(trip)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    gs_all = [(w.groups[gi].rows, w.groups[gi].cols, held[i]) for i, (gi, _, _) in enumerate(share)]
    div_idx = [i for i in range(len(share)) if divided[i]]

    def step():
        for _ in range(w.layers):
            ns.muon_step_host(h, gs_all, [t[1] for t in host], [t[2] for t in host],
                              [t[0] for t in host], w.lr, w.wd, w.mu, w.ns_steps, stream)
            for _ in range(P - 1):
                ns.muon_step_host(h, [gs_all[i] for i in div_idx], [host[i][1] for i in div_idx],
                                  [host[i][2] for i in div_idx], [host[i][0] for i in div_idx],
                                  w.lr, w.wd, w.mu, w.ns_steps, stream)

    steps = max(1, min(args.steps, args.e2e_steps))
    step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    secs = max_over_ranks(time.perf_counter() - t0, world,
                          device=torch.device("cuda", torch.cuda.current_device()))
    nbytes = sum(c * e for c, e in zip(counts, elems)) * 4 * w.layers
    held_gb = sum(hc * e for hc, e in zip(held, elems)) * 12 / 1e9
    del host
    api = "muon_step_host (page-locked host buffers from muon_host_alloc)"
    if P > 1:
        api += (f"; host buffers hold 1/{P} of every group whose count {P} divides "
                f"({held_gb:.1f} GB pinned) and one step is {P} calls, so every step copies "
                "and steps the whole workload")
    return {"value": round(w.matrices * steps / secs, 3), "unit": UNIT,
            "h2d_bytes_per_step": 3 * nbytes, "d2h_bytes_per_step": 2 * nbytes,
            "steps": steps, "ms_per_step": round(secs * 1e3 / steps, 3), "api": api,
            "host_passes": P, "host_pinned_gb": round(held_gb, 2)}


# ----------------------------------------------------------------- CPU oracle
def cpu_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_flops(m: int, n: int, steps: int) -> float:
    """Flops of the oracle's plain iteration on an m x n wide matrix (no
    symmetry: X X^T, A A and B X, 2 m^2 n + 2 m^3 + 2 m^2 n per step)."""
    return steps * (4.0 * m * m * n + 2.0 * m ** 3)


def oracle_shape_seconds(w, per_shape: int, seed_offset: int = 0, shapes=None):
    """Time the oracle on `per_shape` matrices of every distinct wide shape
    of the workload (or of `shapes` only; a tall group costs what its wide
    transpose costs).  Returns ({wide shape: seconds per matrix}, matrices
    timed, seconds)."""
    import numpy as np

    from oracle import muon_oracle as o
    rng = np.random.default_rng(12345 + seed_offset)
    per, done, total = {}, 0, 0.0
    for g in w.groups:
        if g.wide in per or (shapes is not None and g.wide not in shapes):
            continue
        t0 = time.perf_counter()
        for _ in range(per_shape):
            W = (rng.standard_normal((g.rows, g.cols), dtype=np.float32) * np.float32(g.w_std))
            M = (rng.standard_normal((g.rows, g.cols), dtype=np.float32) * np.float32(g.m_std))
            G = (rng.standard_normal((g.rows, g.cols), dtype=np.float32) * np.float32(g.g_std))
            o.muon_step_matrix(W, M, G, lr=w.lr, wd=w.wd, mu=w.mu, ns_steps=w.ns_steps)
        dt = time.perf_counter() - t0
        per[g.wide] = dt / per_shape
        done += per_shape
        total += dt
    return per, done, total


def split_shapes(w, budget: float):
    """Wide shapes the oracle times (one matrix costs at most budget/3 at
    the FP64 rate of one matrix of the cheapest shape) and shapes whose
    time per matrix is extrapolated from the measured rate by their oracle
    flop count.  Returns (timed, extrapolated, probe seconds per matrix)."""
    shapes = sorted(w.wide_batches(), key=lambda s: oracle_flops(s[0], s[1], w.ns_steps))
    cheapest = shapes[0]
    per, _, _ = oracle_shape_seconds(w, 1, 7, shapes={cheapest})
    rate = oracle_flops(*cheapest, w.ns_steps) / max(per[cheapest], 1e-9)
    timed = [s for s in shapes if oracle_flops(*s, w.ns_steps) / rate <= budget / 3.0]
    if cheapest not in timed:
        timed.insert(0, cheapest)
    extra = [s for s in shapes if s not in timed]
    return timed, extra, per[cheapest]


def complete_per_matrix(w, per, extra):
    """Fill in the extrapolated shapes at the FP64 rate the timed shapes
    reached (their flops over their seconds)."""
    fl = sum(oracle_flops(m, n, w.ns_steps) for m, n in per)
    secs = sum(per.values())
    rate = fl / max(secs, 1e-12)
    out = dict(per)
    for m, n in extra:
        out[(m, n)] = oracle_flops(m, n, w.ns_steps) / rate
    return out


def workload_rate(w, per_matrix_seconds) -> float:
    """Matrices per second over the whole workload, each group weighted by
    its matrix count (exact for a single-shape workload)."""
    secs = sum(g.count * per_matrix_seconds[g.wide] for g in w.groups)
    return w.matrices_per_layer / secs


def oracle_sample_text(w, per_shape: int, unit: str, timed, extra) -> str:
    fmt = lambda ss: ", ".join(f"{m}x{n}" for m, n in ss)  # noqa: E731
    text = (f"{per_shape} matrices {unit}of each timed wide shape ({fmt(timed)}) "
            f"of workload {w.name}, FP64 NumPy oracle")
    if extra:
        text += (f"; {fmt(extra)} not timed (one matrix is too long for the sample): time per "
                 "matrix extrapolated from the timed shapes' FP64 rate by the oracle's flop "
                 "count ns_steps*(4 m^2 n + 2 m^3)")
    if len(timed) + len(extra) > 1:
        text += "; rate extrapolated over the workload's group counts"
    return text


def cpu_baseline(w, seconds_budget: float):
    t0 = time.perf_counter()
    timed, extra, probe = split_shapes(w, seconds_budget)
    one = sum(oracle_flops(m, n, w.ns_steps) for m, n in timed) / \
        oracle_flops(*timed[0], w.ns_steps) * probe
    k = int(max(1, min(64, seconds_budget / max(one, 1e-3))))
    per, n, _ = oracle_shape_seconds(w, k, 1, shapes=set(timed))
    full = complete_per_matrix(w, per, extra)
    t = time.perf_counter() - t0
    return {"value": round(workload_rate(w, full), 4), "unit": UNIT, "cores": cpu_cores(),
            "kind": "oracle",
            "sample": oracle_sample_text(w, k, "", timed, extra) + f", {t:.1f} s"}


def run_reference(args, world, rank):
    """The oracle as the reference arm (rank 0 only)."""
    from newton_schulz_03_gb300.workloads import WORKLOADS
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = 10
    # Size one step to a bounded sample so the whole run takes minutes.
    total_budget = 150.0
    per_step_budget = total_budget / (args.steps + args.warmup)
    timed, extra, probe = split_shapes(w, max(per_step_budget, 3.0))
    one = sum(oracle_flops(m, n, w.ns_steps) for m, n in timed) / \
        oracle_flops(*timed[0], w.ns_steps) * probe
    per_step = max(1, int(per_step_budget / max(one, 1e-3)))
    per_step = min(per_step, max(g.count for g in w.groups))
    for i in range(args.warmup):
        oracle_shape_seconds(w, per_step, 100 + i, shapes=set(timed))
    acc = {}
    secs = 0.0
    for i in range(args.steps):
        per, _, t = oracle_shape_seconds(w, per_step, 1000 + i, shapes=set(timed))
        for s_, v in per.items():
            acc[s_] = acc.get(s_, 0.0) + v / args.steps
        secs += t
    value = workload_rate(w, complete_per_matrix(w, acc, extra))
    sample = oracle_sample_text(w, per_step, "per step ", timed, extra)
    return {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w.name, "matrices_per_step_sampled": per_step * len(acc),
                   "note": "CPU oracle on a bounded sample of the workload"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 5 s of steps, 10 to 100; 3 when a step "
                         "takes over 0.6 s)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--max-count", type=int, default=0,
                    help="cap every group's matrix count (small profiling cases)")
    ap.add_argument("--shape", default=None,
                    help="keep only the groups of this wide shape, e.g. 2048x8704 (profiling)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed")
    ap.add_argument("--adamw", action="store_true",
                    help="also measure the AdamW companion kernel (adds an 'adamw' object)")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
