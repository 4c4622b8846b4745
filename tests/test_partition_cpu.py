"""Whole-matrix partition over data-parallel ranks (CPU).

"Frontier Pre-training at Microsoft AI", Method details §5 "Scaling Muon to
16K GPUs", resharding steps 2-3: after the exchange each GPU holds a subset
of complete matrices and orthogonalises them independently.  muon_partition
chooses those subsets: longest processing time first over single matrices,
then one contiguous slice per group and rank.  Checked here without a GPU:
exact cover, the list-scheduling bound, LPT's worst-case ratio against the
optimum found by brute force on small instances, and a world-size-2 gloo
run in which each rank steps its own slices (the CPU oracle stands in for
the per-rank step) and the union equals the one-rank result.
"""

import itertools
import os
import socket

import numpy as np
import pytest

from oracle import muon_oracle as o


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def est_seconds(rows, cols, steps):
    """The partition's documented per-matrix estimate: algorithmic flops at
    1.9 PFLOP/s plus 24 bytes per element at 6.8 TB/s."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (3.0 * m * m * n + m ** 3) / 1.9e15 + 24.0 * m * n / 6.8e12


def check_cover(groups, slices, world):
    for g, (_, _, count) in enumerate(groups):
        got = sorted((first, c) for r in range(world) for gg, first, c in slices[r] if gg == g)
        at = 0
        for first, c in got:
            assert first == at and c > 0
            at += c
        assert at == count, f"group {g}: slices cover {at} of {count}"
    for r in range(world):
        firsts = [s[1] for s in slices[r]]
        assert len({s[0] for s in slices[r]}) == len(slices[r]), "one slice per group and rank"
        assert all(f >= 0 for f in firsts)


def test_partition_covers_every_matrix_once_and_balances(ns):
    rng = np.random.default_rng(11)
    dims = [8, 64, 128, 512, 1536, 2048, 4096, 8704]
    for _ in range(200):
        groups = [(int(rng.choice(dims)), int(rng.choice(dims)), int(rng.choice([0, 1, 3, 17, 512])))
                  for _ in range(int(rng.integers(1, 6)))]
        steps = int(rng.choice([0, 1, 5]))
        world = int(rng.choice([1, 2, 3, 4, 8, 16]))
        slices, secs = ns.muon_partition(groups, world, ns_steps=steps)
        check_cover(groups, slices, world)
        cost = [est_seconds(r, c, steps) for r, c, _ in groups]
        loads = [sum(cost[g] * c for g, _, c in slices[r]) for r in range(world)]
        assert secs == pytest.approx(loads, rel=1e-12, abs=1e-15)
        total = sum(cost[g] * k for g, (_, _, k) in enumerate(groups))
        biggest = max([cost[g] for g, (_, _, k) in enumerate(groups) if k > 0], default=0.0)
        # Every list schedule ends by total/world + the largest item.
        assert max(loads) <= total / world + biggest + 1e-12
        assert max(loads) >= total / world - 1e-12


def test_partition_one_rank_takes_everything(ns):
    groups = [(2048, 8704, 512), (8704, 2048, 512), (8704, 8704, 4)]
    slices, secs = ns.muon_partition(groups, 1)
    assert slices == [[(0, 0, 512), (1, 0, 512), (2, 0, 4)]]
    assert secs[0] == pytest.approx(sum(est_seconds(r, c, 5) * k for r, c, k in groups))


def test_partition_within_lpt_ratio_of_the_optimum(ns):
    """Graham's bound for LPT: makespan <= (4/3 - 1/(3 world)) * optimum,
    the optimum found by trying every assignment of up to 8 matrices."""
    rng = np.random.default_rng(5)
    dims = [64, 256, 512, 1024, 2048]
    for _ in range(60):
        groups = [(int(rng.choice(dims)), int(rng.choice(dims)), int(rng.integers(1, 3)))
                  for _ in range(int(rng.integers(2, 5)))]
        items = [est_seconds(r, c, 5) for r, c, k in groups for _ in range(k)]
        if len(items) > 8:
            continue
        for world in (2, 3):
            _, secs = ns.muon_partition(groups, world)
            best = min(max(sum(t for t, a in zip(items, asg) if a == r) for r in range(world))
                       for asg in itertools.product(range(world), repeat=len(items)))
            assert max(secs) <= (4 / 3 - 1 / (3 * world)) * best * (1 + 1e-12)


def test_partition_rejects_bad_arguments(ns):
    for args in (([(4, 4, 1)], 0), ([(4, 4, 1)], 70000), ([(0, 4, 1)], 2), ([(4, 4, -1)], 2)):
        with pytest.raises(ns.MuonError) as ei:
            ns.muon_partition(*args)
        assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
    with pytest.raises(ns.MuonError):
        ns.muon_partition([(4, 4, 1)], 2, ns_steps=65)


# ------------------------------------------------------------ gloo, 2 ranks
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


GROUPS = [(96, 64, 3), (64, 96, 2), (128, 128, 2), (40, 72, 5)]
HP = dict(lr=0.02, wd=0.1, mu=0.95, ns_steps=5)


def _inputs():
    rng = np.random.default_rng(77)
    return [tuple(rng.standard_normal((k, r, c), dtype=np.float32) for _ in range(3))
            for r, c, k in GROUPS]


def _rank_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import newton_schulz_03_gb300 as pkg
    slices, _ = pkg.muon_partition(GROUPS, world)
    data = _inputs()
    # This rank's step over its own slices only (the oracle stands in for
    # the library's per-rank muon_step on CPU).
    newW = [np.full((k, r, c), np.nan, dtype=np.float32) for r, c, k in GROUPS]
    for g, first, count in slices[rank]:
        W, M, G = data[g]
        for i in range(first, first + count):
            newW[g][i] = o.muon_step_matrix(W[i], M[i], G[i], **HP).W_new
    # Gather every rank's weights; NaN marks matrices a rank did not own.
    flat = torch.from_numpy(np.concatenate([w.ravel() for w in newW]))
    parts = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(parts, flat)
    if rank == 0:
        owned = np.stack([(~torch.isnan(p)).numpy() for p in parts])
        merged = np.where(owned[0], parts[0].numpy(), parts[1].numpy())
        out["owned_once"] = bool((owned.sum(axis=0) == 1).all())
        out["merged"] = merged
    dist.barrier()
    dist.destroy_process_group()


def test_ranks_step_disjoint_slices_whose_union_is_the_one_rank_step(ns):
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_worker, args=(world, port, out), nprocs=world,
                       start_method="spawn", join=True)
    assert out["owned_once"]
    data = _inputs()
    want = np.concatenate([np.stack([o.muon_step_matrix(W[i], M[i], G[i], **HP).W_new
                                     for i in range(W.shape[0])]).ravel()
                           for W, M, G in data])
    assert np.array_equal(out["merged"], want)
