"""GPU parity of the AdamW companion kernel against the FP64 oracle.

Tolerance (derived from the FP32 arithmetic: each of m, v takes two
roundings; the parameter update takes about six on the update term and
one on the decay):
  |dm| <= 1e-6 (|b1 m| + |(1-b1) g|),  |dv| <= 1e-6 (|b2 v| + |(1-b2) g^2|),
  |dp| <= 1e-6 (|p| + |update|)."""

import numpy as np
import pytest

from oracle import muon_oracle as o

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


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


def make(n, rng, offset=0):
    """FP32 tensors of n elements; offset > 0 makes them start 4*offset
    bytes into an allocation (not 16-byte aligned)."""
    out = []
    for scale in (1.0, 1e-2, 1e-2, 1e-4):
        base = torch.empty(n + offset, dtype=torch.float32, device="cuda")
        t = base[offset:]
        vals = rng.standard_normal(n).astype(np.float32) * np.float32(scale)
        if scale == 1e-4:
            vals = np.abs(vals)   # second moment is non-negative
        t.copy_(torch.from_numpy(vals))
        out.append(t)
    return out   # p, g, m, v


def check(before, after, step):
    p0, g0, m0, v0 = (t.cpu().numpy().astype(np.float64) for t in before)
    p1, m1, v1 = (t.cpu().numpy().astype(np.float64) for t in after)
    pr, mr, vr = o.adamw_step(p0.astype(np.float32), g0.astype(np.float32), m0.astype(np.float32),
                              v0.astype(np.float32), step=step, **HP)
    b1, b2 = HP["beta1"], HP["beta2"]
    assert (np.abs(m1 - mr) <= 1e-6 * (np.abs(b1 * m0) + np.abs((1 - b1) * g0)) + 1e-30).all()
    assert (np.abs(v1 - vr) <= 1e-6 * (np.abs(b2 * v0) + np.abs((1 - b2) * g0 * g0)) + 1e-30).all()
    upd = np.abs(pr.astype(np.float64) - p0 * (1 - HP["lr"] * HP["wd"]))
    assert (np.abs(p1 - pr) <= 1e-6 * (np.abs(p0) + upd) + 1e-30).all()


@pytest.mark.parametrize("sizes,offset,step", [
    ([4096], 0, 1), ([1, 7, 4095, 65536 + 3], 0, 3), ([1000, 2048], 1, 10),
    ([0, 333, 0, 2048], 0, 2), ([97] * 45, 0, 5)])
def test_adamw_matches_oracle(ns, h, sizes, offset, step):
    rng = np.random.default_rng(sum(sizes) + offset + step)
    tensors = [make(n, rng, offset) for n in sizes]
    before = [[t.clone() for t in ts] for ts in tensors]
    ns.muon_adamw_step(h, [t[0] for t in tensors], [t[1] for t in tensors],
                       [t[2] for t in tensors], [t[3] for t in tensors], step=step, **HP)
    ns.muon_last_device_error(h)
    for b, a in zip(before, tensors):
        if a[0].numel():
            check(b, [a[0], a[2], a[3]], step)


def test_adamw_bad_arguments(ns, h):
    x = torch.zeros(8, dtype=torch.float32, device="cuda")
    for bad in (dict(HP, beta1=1.0), dict(HP, eps=0.0), dict(HP, lr=float("inf"))):
        with pytest.raises(ns.MuonError):
            ns.muon_adamw_step(h, [x], [x], [x], [x], step=1, **bad)
    with pytest.raises(ns.MuonError):
        ns.muon_adamw_step(h, [x], [x], [x], [x], step=0, **HP)
