"""GPU parity of the method variants (muon_step_ex) against the oracle:
Nesterov momentum, a per-iteration coefficient schedule and the update
scale rules.  Same tolerances as the base step (test_gpu_parity)."""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import ulp_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NS_TOL = 2e-2
LR, WD, MU = 0.02, 0.1, 0.95


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


@pytest.fixture(scope="module")
def h(ns):
    handle = ns.Handle()
    yield handle.value
    handle.close()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_variant(ns, h, shapes, seed, steps=5, **kw):
    rng = np.random.default_rng(seed)
    groups, arrays = [], []
    for r, c, k in shapes:
        groups.append((r, c, k))
        arrays.append(tuple(rng.standard_normal((k, r, c), dtype=np.float32) for _ in range(3)))
    dW = [dev(a[0]) for a in arrays]
    dM = [dev(a[1]) for a in arrays]
    dG = [dev(a[2]) for a in arrays]
    ns.muon_step_ex(h, groups, dM, dG, dW, LR, WD, MU, steps, **kw)
    ns.muon_last_device_error(h)
    return groups, arrays, [t.cpu().numpy() for t in dW], [t.cpu().numpy() for t in dM]


def check(arrays, Wg, Mg, groups, steps, coeffs, nesterov, rule):
    for gi, ((W, M, G), (r, c, k)) in enumerate(zip(arrays, groups)):
        scale = o.update_scale_rule(rule, r, c)
        for i in range(k):
            st = o.muon_step_matrix(W[i], M[i], G[i], lr=LR, wd=WD, mu=MU, ns_steps=steps,
                                    coeffs=coeffs, nesterov=nesterov, update_scale=scale)
            assert ulp_close(Mg[gi][i], st.M_new).all()
            on = np.linalg.norm(st.O)
            dw = np.linalg.norm(Wg[gi][i].astype(np.float64) - st.W_new.astype(np.float64))
            fp = 1e-6 * (np.linalg.norm(W[i]) + LR * scale * on)
            assert (dw - fp) / (LR * scale * on) <= NS_TOL


SHAPES = [(128, 320, 2), (384, 256, 2), (64, 128, 3)]


def test_nesterov(ns, h):
    groups, arrays, Wg, Mg = run_variant(ns, h, SHAPES, 1, nesterov=True)
    check(arrays, Wg, Mg, groups, 5, o.NS_COEFFS, True, o.SCALE_NONE)


def test_coefficient_schedule(ns, h):
    sched = [(4.0848, -6.8946, 2.9270), (3.9505, -6.3029, 2.6377), (3.7418, -5.5913, 2.3037),
             (2.8769, -3.1427, 1.2046), (2.8366, -3.0525, 1.2012)]
    groups, arrays, Wg, Mg = run_variant(ns, h, SHAPES, 2, coeffs=sched)
    check(arrays, Wg, Mg, groups, 5, sched, False, o.SCALE_NONE)


@pytest.mark.parametrize("rule", [1, 2])
def test_scale_rules(ns, h, rule):
    groups, arrays, Wg, Mg = run_variant(ns, h, SHAPES, 3 + rule, scale_rule=rule)
    check(arrays, Wg, Mg, groups, 5, o.NS_COEFFS, False, rule)


def test_defaults_equal_muon_step(ns, h):
    rng = np.random.default_rng(9)
    W, M, G = (rng.standard_normal((3, 256, 512), dtype=np.float32) for _ in range(3))
    a = [dev(W), dev(M), dev(G)]
    b = [dev(W), dev(M), dev(G)]
    ns.muon_step(h, [(256, 512, 3)], [a[1]], [a[2]], [a[0]], LR, WD, MU, 5)
    ns.muon_step_ex(h, [(256, 512, 3)], [b[1]], [b[2]], [b[0]], LR, WD, MU, 5)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_options_rejected(ns, h):
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(ns.MuonError):
        ns.muon_step_ex(h, [(8, 8, 1)], [x], [x], [x], LR, WD, MU, 5, scale_rule=7)
    with pytest.raises(ns.MuonError):
        ns.muon_step_ex(h, [(8, 8, 1)], [x], [x], [x], LR, WD, MU, 2,
                        coeffs=[(1.0, 2.0, float("nan")), (1.0, 1.0, 1.0)])
