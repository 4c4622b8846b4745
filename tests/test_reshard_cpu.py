"""The resharded Muon step on CPU ranks (gloo).

"Frontier Pre-training at Microsoft AI", Method details §5, resharding
steps 1-5, and the replicated router weights of its tuning bullets.  The
exchange layout (ZeRO shards, owners from muon_partition) and the two
all-to-alls run exactly as on GPUs; the local compute between them is the
CPU oracle (FP64 payloads), so the composed step must equal the oracle's
one-rank step matrix by matrix, and an identity in place of the
Newton-Schulz step must return every shard its own BF16 momentum bit for
bit (shard -> whole -> shard).
"""

import os
import socket

import numpy as np
import pytest

from oracle import muon_oracle as o

torch = pytest.importorskip("torch")

GROUPS = [(64, 32, 3, 1.0), (32, 64, 5, 0.5), (48, 40, 2, 1.0), (16, 32, 2, 1.0), (40, 8, 7, 2.0)]
REPLICATED = (3,)            # a router-like group, held whole by every rank
HP = dict(lr=0.02, wd=0.1, mu=0.95)
STEPS = 5


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def _data():
    rng = np.random.default_rng(2025)
    return [tuple(rng.standard_normal((k, r, c), dtype=np.float32) * np.float32(s)
                  for s in (0.02, 1e-3, 1e-3)) for r, c, k, _ in GROUPS]


class OracleOps:
    """The oracle as the local compute (CPU, FP64 payloads)."""

    def empty(self, n, dtype, like):
        return torch.empty(n, dtype=dtype)

    def zeros(self, shape, dtype, like):
        return torch.zeros(shape, dtype=dtype)

    def shard_cast(self, M, G, mu, begin, end, E):
        Mn = o.momentum_update(M.numpy(), G.numpy(), mu)
        M.copy_(torch.from_numpy(Mn))
        X = torch.from_numpy(o.bf16_rne(Mn))
        k0, k1 = begin // E, ((end - 1) // E + 1 if end > begin else begin // E)
        sums = []
        for k in range(k0, k1):
            lo, hi = max(begin, k * E) - begin, min(end, (k + 1) * E) - begin
            piece = Mn[lo:hi].astype(np.float64)
            sums.append(float(np.sum(piece * piece)))
        return X, torch.tensor(sums, dtype=torch.float64)

    def orthogonalise(self, X, sums, rows, cols, steps):
        out = torch.empty((X.shape[0], rows, cols), dtype=torch.float64)
        for k in range(X.shape[0]):
            Xw, tr = o.to_wide(X[k].numpy())
            s = float(np.sqrt(sums[k].numpy().sum())) + o.NORM_EPS
            Ow = o.newton_schulz(Xw, s, steps)
            out[k] = torch.from_numpy(np.ascontiguousarray(Ow.T if tr else Ow))
        return out

    def apply(self, W, O, lr, wd, scale):
        W.copy_(torch.from_numpy(o.apply_update(W.numpy(), O.numpy(), lr, wd, scale)))


class IdentityOps(OracleOps):
    """Newton-Schulz replaced by the identity and the apply by a copy: the
    update a shard gets back is the BF16 momentum it sent out."""

    def orthogonalise(self, X, sums, rows, cols, steps):
        return X.clone()

    def apply(self, W, O, lr, wd, scale):
        W.copy_(O.to(W.dtype))


def _shards(plan, rank, data):
    state = []
    for g, gl in enumerate(plan.groups):
        b, e = gl.shard[rank]
        trip = tuple(torch.from_numpy(a.reshape(-1)[b:e].copy()) for a in data[g])
        state.append((trip[1], trip[2], trip[0]))   # (M, G, W)
    return state


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, mode, out, overlap=True):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from newton_schulz_03_gb300.reshard import ReshardPlan, resharded_step
    plan = ReshardPlan(GROUPS, world, replicated=REPLICATED, ns_steps=STEPS)
    state = _shards(plan, rank, _data())
    ops = OracleOps() if mode == "oracle" else IdentityOps()
    resharded_step(plan, rank, state, HP["lr"], HP["wd"], HP["mu"], ops, overlap=overlap)
    out[rank] = [(M.numpy().copy(), W.numpy().copy()) for M, _, W in state]
    dist.barrier()
    dist.destroy_process_group()


def _run(world, mode, overlap=True):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), mode, out, overlap), nprocs=world,
                       start_method="spawn", join=True)
    return dict(out)


def _merge(ns, world, got, g):
    """The group's flat (M, W) from the ranks' shards (a replicated group:
    rank 0's copy, after checking every rank holds the same)."""
    from newton_schulz_03_gb300.reshard import ReshardPlan
    plan = ReshardPlan(GROUPS, world, replicated=REPLICATED, ns_steps=STEPS)
    gl = plan.groups[g]
    if gl.replicated:
        for r in range(1, world):
            assert np.array_equal(got[r][g][1], got[0][g][1])
        return got[0][g]
    return tuple(np.concatenate([got[r][g][i] for r in range(world)]) for i in (0, 1))


@pytest.mark.parametrize("world,overlap", [(2, True), (3, True), (2, False)])
def test_resharded_step_equals_the_one_rank_oracle_step(ns, world, overlap):
    # overlap: exchanges started asynchronously (one group's collectives
    # beside another group's Newton-Schulz step); else one after the other.
    got = _run(world, "oracle", overlap)
    data = _data()
    for g, (r, c, k, scale) in enumerate(GROUPS):
        M, W = _merge(ns, world, got, g)
        Wd, Md, Gd = data[g]
        for i in range(k):
            ref = o.muon_step_matrix(Wd[i], Md[i], Gd[i], ns_steps=STEPS, update_scale=scale,
                                     **HP)
            Mi = M[i * r * c:(i + 1) * r * c].reshape(r, c)
            Wi = W[i * r * c:(i + 1) * r * c].reshape(r, c)
            assert np.array_equal(Mi, ref.M_new), f"group {g} matrix {i}: momentum"
            # Only the norm's summation order differs (pieces vs whole).
            assert np.allclose(Wi, ref.W_new, rtol=0, atol=1e-6 * np.abs(ref.W_new).max()), \
                f"group {g} matrix {i}: weights"


def test_shard_whole_shard_round_trip_is_exact(ns):
    world = 3
    got = _run(world, "identity")
    data = _data()
    for g, (r, c, k, _) in enumerate(GROUPS):
        _, W = _merge(ns, world, got, g)
        Wd, Md, Gd = data[g]
        Mn = o.momentum_update(Md.reshape(-1), Gd.reshape(-1), HP["mu"])
        assert np.array_equal(W, o.bf16_rne(Mn).astype(np.float32)), f"group {g}"


def test_exchange_layout_is_consistent(ns):
    from newton_schulz_03_gb300.reshard import ReshardPlan
    for world in (1, 2, 3, 8):
        plan = ReshardPlan(GROUPS + [(2048, 8704, 512), (8704, 2048, 512)], world,
                           replicated=REPLICATED)
        for gl in plan.groups:
            E = gl.elems
            assert sum(c for _, c in gl.own) == gl.count
            if gl.replicated:
                continue
            covered = 0
            for q, (b, e) in enumerate(gl.shard):
                assert b == covered or e == b
                covered = max(covered, e)
                assert sum(gl.send[q]) == e - b              # every element goes to one owner
            assert covered == gl.total
            for p, (f, c) in enumerate(gl.own):
                assert sum(gl.send[q][p] for q in range(world)) == c * E
