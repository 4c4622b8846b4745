"""The step can be captured in a CUDA graph and replayed: after one
ordinary call (which allocates the workspace and caches the plan), a
muon_step enqueues only kernel launches, so a captured step replays the
same computation bit for bit."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


@pytest.mark.parametrize("shapes", [[(384, 256, 3), (128, 64, 4)], [(1024, 1024, 2)]])
def test_graph_replay_equals_eager(ns, shapes):
    rng = np.random.default_rng(5)
    groups = [tuple(s) for s in shapes]
    host = [tuple(rng.standard_normal((k, r, c), dtype=np.float32) for _ in range(3))
            for r, c, k in groups]

    def state():
        return [[torch.from_numpy(a.copy()).cuda() for a in t] for t in host]

    eager, cap = state(), state()
    with ns.Handle() as h:
        args = lambda st: ([t[1] for t in st], [t[2] for t in st], [t[0] for t in st])
        # Eager reference: two steps.
        for _ in range(2):
            ns.muon_step(h.value, groups, *args(eager), 0.02, 0.1, 0.95, 5)
        # One ordinary call on scratch copies sets up workspace and plan.
        warm = state()
        ns.muon_step(h.value, groups, *args(warm), 0.02, 0.1, 0.95, 5)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=s):
            ns.muon_step(h.value, groups, *args(cap), 0.02, 0.1, 0.95, 5)
        # Capturing runs nothing: replay twice = two steps.
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        ns.muon_last_device_error(h.value)
    for a, b in zip(eager, cap):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
