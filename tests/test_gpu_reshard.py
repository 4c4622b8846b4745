"""The resharded step's kernels on the GPU, and the composed step with them.

Unit checks of the shard-side entry points against the oracle and the
one-GPU kernels, then the whole resharded step ("Frontier Pre-training at
Microsoft AI", Method details §5, resharding steps 1-5) with the library
as the local compute: the ranks run as threads of one process on one GPU,
each with its own handle, and exchange through a host-side stand-in for
the collectives (device copies between the threads' buffers after a host
barrier).  No kernel waits on another rank's kernel.  The result must match
the one-GPU muon_step: momenta bit for bit, weights within the
Newton-Schulz tolerance (the norm is summed from shard pieces in another
order).
"""

import threading

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import u16, ulp_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def test_shard_cast_matches_the_oracle(ns):
    rng = np.random.default_rng(3)
    E, count = 96 * 40, 9
    M = rng.standard_normal(count * E, dtype=np.float32)
    G = rng.standard_normal(count * E, dtype=np.float32)
    b, e = 1234, 7 * E + 77                      # cuts matrices 0 and 7
    dM = torch.from_numpy(M[b:e].copy()).cuda()
    dG = torch.from_numpy(G[b:e].copy()).cuda()
    X = torch.empty(e - b, dtype=torch.int16, device="cuda")
    sums = torch.empty(8, dtype=torch.float32, device="cuda")
    with ns.Handle() as h:
        ns.muon_shard_momentum_cast(h.value, b, e, E, dM, dG, 0.95, X, sums)
        ns.muon_last_device_error(h.value)
    Mn = o.momentum_update(M[b:e], G[b:e], 0.95)
    assert ulp_close(dM.cpu().numpy(), Mn).all()
    assert np.array_equal(u16(X), o.bf16_rne_bits(dM.cpu().numpy()))
    Mg = dM.cpu().numpy().astype(np.float64)
    for y, k in enumerate(range(b // E, (e - 1) // E + 1)):
        lo, hi = max(b, k * E) - b, min(e, (k + 1) * E) - b
        want = np.sum(Mg[lo:hi] ** 2)
        assert abs(float(sums[y]) - want) <= 1e-5 * want


def test_transpose_norm_and_shard_apply(ns):
    rng = np.random.default_rng(4)
    rows, cols, count = 200, 72, 3
    src = o.bf16_rne_bits(rng.standard_normal((count, rows, cols), dtype=np.float32))
    dsrc = torch.from_numpy(src.view(np.int16)).cuda()
    dst = torch.empty((count, cols, rows), dtype=torch.int16, device="cuda")
    W = rng.standard_normal((count, cols, rows), dtype=np.float32)
    dW1 = torch.from_numpy(W.copy()).cuda()
    dW2 = torch.from_numpy(W.copy()).cuda()
    sumsq = torch.from_numpy(np.abs(rng.standard_normal((count, 3), dtype=np.float32))).cuda()
    inv = torch.empty(count, dtype=torch.float32, device="cuda")
    with ns.Handle() as h:
        ns.muon_transpose_bf16(h.value, rows, cols, count, dsrc, dst)
        ns.muon_norm_from_sumsq(h.value, cols, rows, count, 3, sumsq, dst, inv)
        # The flat shard apply and the one-GPU apply of a wide matrix share
        # their arithmetic: same bits.
        ns.muon_shard_apply(h.value, dW1.numel(), dW1, dst, 0.02, 0.1, 1.5)
        ns.muon_apply_update(h.value, cols, rows, count, dW2, dst, 0.02, 0.1, 1.5)
        ns.muon_last_device_error(h.value)
    assert np.array_equal(u16(dst), np.swapaxes(src, 1, 2))
    want = 1.0 / (np.sqrt(sumsq.cpu().numpy().astype(np.float64).sum(axis=1)) + o.NORM_EPS)
    assert np.allclose(inv.cpu().numpy(), want, rtol=1e-6, atol=0)
    assert torch.equal(dW1, dW2)
    ref = o.apply_update(W, o.bf16_bits_to_f64(np.swapaxes(src, 1, 2)), 0.02, 0.1, 1.5)
    assert np.allclose(dW1.cpu().numpy(), ref, rtol=1e-6, atol=1e-7)


class ThreadComm:
    """Host-side stand-in for the collectives between rank threads of one
    process: every thread posts its send buffer, waits at a barrier, copies
    the pieces addressed to it, synchronises and waits again."""

    def __init__(self, world):
        self.world = world
        self.bar = threading.Barrier(world, timeout=120)
        self.slots = [None] * world
        self.local = threading.local()

    class _Done:
        def wait(self):
            return None

    def all_to_all(self, out, inp, out_splits, in_splits, async_op=False):
        r = self.local.rank
        self.slots[r] = (inp, list(in_splits))
        self.bar.wait()
        at = 0
        for q in range(self.world):
            qin, qs = self.slots[q]
            off, n = sum(qs[:r]), qs[r]
            if n:
                out[at:at + n].copy_(qin[off:off + n])
            at += n
        torch.cuda.synchronize()
        self.bar.wait()
        return self._Done()

    def all_gather(self, out_list, inp, async_op=False):
        r = self.local.rank
        self.slots[r] = (inp, None)
        self.bar.wait()
        for q in range(self.world):
            out_list[q].copy_(self.slots[q][0])
        torch.cuda.synchronize()
        self.bar.wait()
        return self._Done()


GROUPS = [(256, 128, 3, 1.0), (128, 256, 5, 0.5), (512, 512, 2, 1.0), (64, 256, 2, 1.0),
          (136, 64, 7, 2.0)]
REPLICATED = (3,)
HP = dict(lr=0.02, wd=0.1, mu=0.95)


@pytest.mark.parametrize("world", [2, 3])
def test_resharded_step_with_the_library_matches_the_one_gpu_step(ns, world):
    from newton_schulz_03_gb300.reshard import LibraryOps, ReshardPlan, resharded_step
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    full = [tuple(torch.randn((k, r, c), generator=gen, device="cuda") * s
                  for s in (0.02, 1e-3, 1e-3)) for r, c, k, _ in GROUPS]
    plan = ReshardPlan(GROUPS, world, replicated=REPLICATED)
    states = []
    for rank in range(world):
        st = []
        for g, gl in enumerate(plan.groups):
            b, e = gl.shard[rank]
            W, M, G = (t.reshape(-1)[b:e].clone() for t in full[g])
            st.append((M, G, W))
        states.append(st)
    single = [tuple(t.clone() for t in trip) for trip in full]
    handles = [ns.Handle() for _ in range(world)]
    # One-GPU step first (also sets up the kernels' cached launch state).
    ns.muon_step(handles[0].value, [g[:4] for g in GROUPS], [t[1] for t in single],
                 [t[2] for t in single], [t[0] for t in single], HP["lr"], HP["wd"], HP["mu"], 5)
    ns.muon_last_device_error(handles[0].value)
    torch.cuda.synchronize()
    comm = ThreadComm(world)
    errors = []

    def run(rank):
        try:
            comm.local.rank = rank
            resharded_step(plan, rank, states[rank], HP["lr"], HP["wd"], HP["mu"],
                           LibraryOps(handles[rank].value), comm)
            torch.cuda.synchronize()
            ns.muon_last_device_error(handles[rank].value)
        except BaseException as exc:   # noqa: BLE001 -- reported below
            errors.append(exc)
            comm.bar.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    for h in handles:
        h.close()
    assert not errors, errors
    for g, (r, c, k, scale) in enumerate(GROUPS):
        gl = plan.groups[g]
        if gl.replicated:
            parts = [states[q][g] for q in range(world)]
            for q in range(1, world):
                assert torch.equal(parts[q][2], parts[0][2])
            M, W = parts[0][0], parts[0][2]
        else:
            M = torch.cat([states[q][g][0] for q in range(world)])
            W = torch.cat([states[q][g][2] for q in range(world)])
        Ms, Ws = single[g][1].reshape(-1), single[g][0].reshape(-1)
        assert torch.equal(M, Ms), f"group {g}: momenta differ"
        W0 = full[g][0].reshape(-1)
        for i in range(k):
            sl = slice(i * r * c, (i + 1) * r * c)
            step_single = (W0[sl].double() * (1 - HP["lr"] * HP["wd"]) - Ws[sl].double())
            diff = (W[sl].double() - Ws[sl].double()).norm().item()
            assert diff <= 1e-2 * step_single.norm().item() + 1e-7, f"group {g} matrix {i}"


def test_resharded_step_at_full_size_matches_the_one_gpu_step(ns):
    """The L=48 expert workload (1024 matrices, 77 GB of FP32 state) over
    two thread ranks: each rank's shard of a group holds 1.6e9 elements and
    rank 1's shard spans global offsets up to 3.2e9 (beyond 2^31, in the
    shard kernels' piece arithmetic), and the exchanges move whole
    1536 x 4096 matrices.  Sampled matrices: momenta bit for bit, weights
    within 1% of the update, against muon_step on the same data."""
    from newton_schulz_03_gb300.reshard import LibraryOps, ReshardPlan, resharded_step
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_torch
    w = WORKLOADS["l48_experts"]
    free, _ = torch.cuda.mem_get_info()
    need = sum(g.numel for g in w.groups) * (12 + 12 + 12) + (16 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on the device")
    world = 2
    groups = [(g.rows, g.cols, g.count) for g in w.groups]
    plan = ReshardPlan(groups, world, ns_steps=w.ns_steps)
    full = [make_group_torch(w, gi, "cuda") for gi in range(len(w.groups))]
    samples = [(0, 0), (0, 7), (0, 300), (1, 511), (1, 256)]
    W0 = {k: full[k[0]][0][k[1]].clone() for k in samples}
    states = []
    for rank in range(world):
        st = []
        for g, gl in enumerate(plan.groups):
            b, e = gl.shard[rank]
            W, M, G = (t.reshape(-1)[b:e].clone() for t in full[g])
            st.append((M, G, W))
        states.append(st)
    handles = [ns.Handle() for _ in range(world)]
    ns.muon_step(handles[0].value, groups, [t[1] for t in full], [t[2] for t in full],
                 [t[0] for t in full], w.lr, w.wd, w.mu, w.ns_steps)
    ns.muon_last_device_error(handles[0].value)
    torch.cuda.synchronize()
    comm = ThreadComm(world)
    errors = []

    def run(rank):
        try:
            comm.local.rank = rank
            resharded_step(plan, rank, states[rank], w.lr, w.wd, w.mu,
                           LibraryOps(handles[rank].value), comm)
            torch.cuda.synchronize()
            ns.muon_last_device_error(handles[rank].value)
        except BaseException as exc:   # noqa: BLE001 -- reported below
            errors.append(exc)
            comm.bar.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    for h in handles:
        h.close()
    assert not errors, errors
    for gi, i in samples:
        gl = plan.groups[gi]
        E = gl.elems
        lo = i * E
        M = torch.cat([states[q][gi][0] for q in range(world)])[lo:lo + E]
        W = torch.cat([states[q][gi][2] for q in range(world)])[lo:lo + E]
        assert torch.equal(M, full[gi][1][i].reshape(-1)), f"group {gi} matrix {i}: momentum"
        Ws = full[gi][0][i].reshape(-1).double()
        step = W0[(gi, i)].reshape(-1).double() * (1 - w.lr * w.wd) - Ws
        diff = (W.double() - Ws).norm().item()
        assert diff <= 1e-2 * step.norm().item() + 1e-7, f"group {gi} matrix {i}: weights"
    del full, states
    torch.cuda.empty_cache()
