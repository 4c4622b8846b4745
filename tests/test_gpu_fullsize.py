"""Full-size parity: the workloads at their real sizes, in the launch
configuration the benchmark times (one muon_step over every group of the
workload), checked on sampled matrices against the CPU oracle.

Every configured shape meets the FP64 oracle here, the largest ones
included: an 8704 x 8704 attention projection and the 8704 x 13056 shared
expert of the L=102 layer take the oracle about a minute each on the host
cores.
"""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import ulp_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NS_TOL = 2e-2


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def free_bytes():
    free, _ = torch.cuda.mem_get_info()
    return free


def step_workload(ns, wname, samples):
    """Step a whole workload once on device-generated inputs; return the
    sampled matrices' inputs and outputs on the host."""
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_torch
    w = WORKLOADS[wname]
    need = sum(g.numel for g in w.groups) * 12 + (9 << 30)
    if free_bytes() < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on the device")
    groups = [(g.rows, g.cols, g.count) for g in w.groups]
    tensors = [make_group_torch(w, gi, "cuda") for gi in range(len(w.groups))]
    before = {(gi, i): tuple(t[i].cpu().numpy() for t in tensors[gi])
              for gi, i in samples}
    Ws, Ms, Gs = ([t[k] for t in tensors] for k in range(3))
    with ns.Handle() as h:
        ns.muon_step(h.value, groups, Ms, Gs, Ws, w.lr, w.wd, w.mu, w.ns_steps)
        ns.muon_last_device_error(h.value)
    after = {(gi, i): (Ws[gi][i].cpu().numpy(), Ms[gi][i].cpu().numpy())
             for gi, i in samples}
    del tensors, Ws, Ms, Gs
    torch.cuda.empty_cache()
    return w, before, after


def check_sample(w, before, after, key, model=False):
    """Oracle check of one sampled matrix; with `model`, also the error
    model: the update's error must match that of the oracle's BF16
    emulation (rounding where the kernels store) within 15% + 5e-4."""
    gi, i = key
    W, M, G = before[key]
    Wg, Mg = after[key]
    st = o.muon_step_matrix(W, M, G, lr=w.lr, wd=w.wd, mu=w.mu, ns_steps=w.ns_steps)
    assert ulp_close(Mg, st.M_new).all()
    on = np.linalg.norm(st.O)
    dw = np.linalg.norm(Wg.astype(np.float64) - st.W_new.astype(np.float64))
    fp = 1e-6 * (np.linalg.norm(W) + w.lr * on)
    if on == 0.0:
        assert dw <= fp, "zero momentum must only decay the weights"
        return 0.0
    err = (dw - fp) / (w.lr * on)
    assert err <= NS_TOL, f"group {gi} matrix {i}: update error {err:.3e}"
    if model:
        emu = o.muon_step_matrix(W, M, G, lr=w.lr, wd=w.wd, mu=w.mu, ns_steps=w.ns_steps,
                                 emulate_bf16=True)
        bound = 1.15 * np.linalg.norm(emu.O - st.O) / on + 5e-4
        assert err <= bound, f"group {gi} matrix {i}: {err:.3e} vs error model {bound:.3e}"
    return err


def test_fullsize_l24_attention(ns):
    # 96 x 2048^2 (rung L=24 attention).
    w, before, after = step_workload(ns, "l24_attention", [(0, 0), (0, 57), (0, 95)])
    for k in before:
        check_sample(w, before, after, k, model=(k == (0, 0)))


def test_fullsize_l48_experts(ns):
    # 1024 matrices: up (1536 x 4096) and down (4096 x 1536, transposed);
    # matrix 7 of each group has zero gradient and momentum.
    samples = [(0, 0), (0, 7), (1, 7), (1, 300), (0, 511)]
    w, before, after = step_workload(ns, "l48_experts", samples)
    for k in samples:
        check_sample(w, before, after, k, model=(k in ((0, 0), (1, 300))))


def test_fullsize_l48_model_layer(ns):
    # One resident layer of the whole-model step: attention, shared expert,
    # routed experts and the router in one call.
    samples = [(0, 3), (1, 0), (2, 0), (3, 100), (4, 511), (5, 0)]
    w, before, after = step_workload(ns, "l48_model", samples)
    for k in samples:
        check_sample(w, before, after, k)


def test_fullsize_l102_layer(ns):
    # 226 GB of FP32 state.  Experts of both orientations, the shared
    # expert's tall 13056 x 8704 up-projection and an 8704 x 8704 attention
    # projection against the FP64 oracle; those two and a transposed expert
    # also against the error model.
    samples = [(0, 0), (1, 511), (0, 7), (2, 0), (4, 3)]
    w, before, after = step_workload(ns, "l102_layer", samples)
    for k in samples:
        check_sample(w, before, after, k, model=(k in ((2, 0), (4, 3), (1, 511))))


def test_fullsize_l48_experts_variants(ns):
    """The expert workload at full size through muon_step_ex with Nesterov
    momentum, a per-iteration coefficient schedule and the RMS-matching
    update scale, on sampled matrices of both orientations."""
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_torch
    w = WORKLOADS["l48_experts"]
    need = sum(g.numel for g in w.groups) * 12 + (9 << 30)
    if free_bytes() < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on the device")
    sched = [(4.0848, -6.8946, 2.9270), (3.9505, -6.3029, 2.6377), (3.7418, -5.5913, 2.3037),
             (2.8769, -3.1427, 1.2046), (2.8366, -3.0525, 1.2012)]
    samples = [(0, 3), (1, 400)]
    groups = [(g.rows, g.cols, g.count) for g in w.groups]
    tensors = [make_group_torch(w, gi, "cuda") for gi in range(len(w.groups))]
    before = {k: tuple(t[k[1]].cpu().numpy() for t in tensors[k[0]]) for k in samples}
    Ws, Ms, Gs = ([t[k] for t in tensors] for k in range(3))
    with ns.Handle() as h:
        ns.muon_step_ex(h.value, groups, Ms, Gs, Ws, w.lr, w.wd, w.mu, 5, nesterov=True,
                        coeffs=sched, scale_rule=ns.SCALE_RMS_MATCH)
        ns.muon_last_device_error(h.value)
    after = {k: (Ws[k[0]][k[1]].cpu().numpy(), Ms[k[0]][k[1]].cpu().numpy()) for k in samples}
    del tensors, Ws, Ms, Gs
    torch.cuda.empty_cache()
    for (gi, i) in samples:
        W, M, G = before[(gi, i)]
        Wg, Mg = after[(gi, i)]
        g = w.groups[gi]
        scale = o.update_scale_rule(o.SCALE_RMS_MATCH, g.rows, g.cols)
        kw = dict(lr=w.lr, wd=w.wd, mu=w.mu, ns_steps=5, coeffs=sched, nesterov=True,
                  update_scale=scale)
        st = o.muon_step_matrix(W, M, G, **kw)
        assert ulp_close(Mg, st.M_new).all()
        on = np.linalg.norm(st.O)
        dw = np.linalg.norm(Wg.astype(np.float64) - st.W_new.astype(np.float64))
        fp = 1e-6 * (np.linalg.norm(W) + w.lr * scale * on)
        err = (dw - fp) / (w.lr * scale * on)
        assert err <= NS_TOL, f"group {gi} matrix {i}: update error {err:.3e}"
        emu = o.muon_step_matrix(W, M, G, emulate_bf16=True, **kw)
        bound = 1.15 * np.linalg.norm(emu.O - st.O) / on + 5e-4
        assert err <= bound, f"group {gi} matrix {i}: {err:.3e} vs error model {bound:.3e}"


@pytest.mark.parametrize("pinning", ["torch", "muon_host_alloc"])
def test_fullsize_l24_host_buffers_match_device_step(ns, pinning):
    """The end-to-end entry point at a benchmark size: muon_step_host on
    pinned host buffers (pipelined pieces, ramped first and last pieces)
    gives the device-buffer step's weights and momenta bit for bit, with
    torch's pinned memory and with the library's own page-locked
    allocation."""
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_torch
    w = WORKLOADS["l24_attention"]
    need = sum(g.numel for g in w.groups) * 12 + (9 << 30)
    if free_bytes() < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on the device")
    groups = [(g.rows, g.cols, g.count) for g in w.groups]
    W, M, G = make_group_torch(w, 0, "cuda")
    if pinning == "torch":
        Wh, Mh, Gh = (t.cpu().pin_memory() for t in (W, M, G))
    else:
        Wh, Mh, Gh = (ns.host_empty(tuple(t.shape)) for t in (W, M, G))
        for hst, dev in zip((Wh, Mh, Gh), (W, M, G)):
            hst.copy_(dev)
    with ns.Handle() as h:
        ns.muon_step_host(h.value, groups, [Mh], [Gh], [Wh], w.lr, w.wd, w.mu, w.ns_steps)
        ns.muon_step(h.value, groups, [M], [G], [W], w.lr, w.wd, w.mu, w.ns_steps)
        ns.muon_last_device_error(h.value)
    assert torch.equal(Mh, M.cpu())
    assert torch.equal(Wh, W.cpu())
    del W, M, G, Wh, Mh, Gh
    torch.cuda.empty_cache()
