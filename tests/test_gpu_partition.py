"""The whole-matrix partition on the GPU: stepping each rank's share of a
group list on its own gives, matrix for matrix, the bits of the one-rank
step ("Frontier Pre-training at Microsoft AI", Method details §5, resharding
steps 2-3: each GPU orthogonalises the complete matrices it holds, with no
dependence on the others).  One GPU runs the ranks' shares one after the
other; nothing waits on another rank."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

GROUPS = [(256, 512, 7), (512, 256, 5), (1024, 1024, 3), (64, 128, 9), (130, 72, 4),
          (2048, 8704, 2)]
HP = dict(lr=0.02, wd=0.1, mu=0.95, ns_steps=5)


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def _state(seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    return [tuple(torch.randn((k, r, c), generator=gen, device="cuda") * s
                  for s in (0.02, 1e-3, 1e-3)) for r, c, k in GROUPS]


@pytest.mark.parametrize("world", [2, 3, 8])
def test_rank_shares_reproduce_the_one_rank_step(ns, world):
    whole = _state(5)
    parts = [tuple(t.clone() for t in trip) for trip in whole]
    with ns.Handle() as h:
        ns.muon_step(h.value, GROUPS, [t[1] for t in whole], [t[2] for t in whole],
                     [t[0] for t in whole], HP["lr"], HP["wd"], HP["mu"], HP["ns_steps"])
        slices, secs = ns.muon_partition(GROUPS, world, HP["ns_steps"])
        assert len(secs) == world
        for rank in range(world):
            if not slices[rank]:
                continue
            gs = [(GROUPS[g][0], GROUPS[g][1], c) for g, _, c in slices[rank]]
            W = [parts[g][0][f:f + c] for g, f, c in slices[rank]]
            M = [parts[g][1][f:f + c] for g, f, c in slices[rank]]
            G = [parts[g][2][f:f + c] for g, f, c in slices[rank]]
            ns.muon_step(h.value, gs, M, G, W, HP["lr"], HP["wd"], HP["mu"], HP["ns_steps"])
        ns.muon_last_device_error(h.value)
    torch.cuda.synchronize()
    for gi in range(len(GROUPS)):
        assert torch.equal(parts[gi][0], whole[gi][0]), f"group {gi}: weights differ"
        assert torch.equal(parts[gi][1], whole[gi][1]), f"group {gi}: momenta differ"
    # Every matrix was stepped exactly once: the weights moved everywhere.
    assert all(bool(np.all((parts[gi][0] != _state(5)[gi][0]).any(dim=(1, 2)).cpu().numpy()))
               for gi in range(len(GROUPS)))
