"""GPU parity: every step of the CUDA path against the CPU oracle.

Tolerances:
* momentum update: within 1 FP32 ulp of the oracle (the GPU's fused
  multiply-add rounds once; the oracle's FP64 sum rounds twice at most);
* BF16 cast: bit-exact (both sides round the same FP32 values);
* norm: 1e-6 relative;
* weight update: |dW| <= 1e-6 (|W| + |lr s O|) elementwise, given the same
  BF16 update O on both sides (bound derived from four FP32 roundings);
* Newton-Schulz: relative Frobenius error <= 2e-2 per matrix against the
  FP64 oracle (BF16 operands, FP32 accumulation) for matrices with at least
  64 rows after the transpose to wide (every configured shape).  Smaller
  edge-case matrices get 4e-2: rounding to BF16 at exactly the GPU's
  points, in FP64 otherwise, already errs by up to 3.1e-2 on 5 x 37
  matrices (200 seeds), so 2e-2 is below the format's floor there.
Sizes span several 128-row tiles and ragged tails.
"""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import rel_fro, to_wide, u16, ulp_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NS_TOL = 2e-2
NS_TOL_SMALL = 4e-2


def ns_tol(rows, cols):
    return NS_TOL if min(rows, cols) >= 64 else NS_TOL_SMALL


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


# ----------------------------------------------------------------- step 1
@pytest.mark.parametrize("rows,cols,count", [
    (128, 64, 4), (64, 128, 3), (200, 136, 2), (72, 300, 2), (1, 40, 3), (37, 5, 2),
    (256, 256, 1), (130, 7, 2), (64, 64, 0)])
def test_momentum_cast(ns, h, rows, cols, count):
    rng = np.random.default_rng(rows * 1000 + cols + count)
    M = rng.standard_normal((count, rows, cols), dtype=np.float32)
    G = rng.standard_normal((count, rows, cols), dtype=np.float32)
    mu = 0.95
    m, n = min(rows, cols), max(rows, cols)
    dM, dG = dev(M), dev(G)
    X = torch.zeros((max(count, 1), m, n), dtype=torch.int16, device="cuda")
    inv = torch.zeros(max(count, 1), dtype=torch.float32, device="cuda")
    ns.muon_momentum_cast(h, rows, cols, count, dM, dG, mu, X, inv)
    ns.muon_last_device_error(h)
    if count == 0:
        return
    Mg = dM.cpu().numpy()
    ref = o.momentum_update(M, G, mu)
    assert ulp_close(Mg, ref).all()
    # Cast: bit-exact against the oracle's RNE of the GPU's own FP32 values.
    want_bits = o.bf16_rne_bits(to_wide(Mg))
    np.testing.assert_array_equal(u16(X)[:count], want_bits)
    for i in range(count):
        s = o.frobenius_scale(Mg[i])
        assert abs(inv.cpu().numpy()[i] * s - 1.0) < 1e-6


# ----------------------------------------------------------------- step 5
@pytest.mark.parametrize("rows,cols,count", [
    (128, 64, 4), (64, 128, 3), (200, 136, 2), (37, 5, 2), (1, 40, 3), (130, 7, 2),
    # tall, double-buffered kernel: ragged last row tile (partial 16-byte
    # runs), several tiles per block of the resident grid
    (1000, 132, 3), (520, 64, 5), (4096, 1536, 2), (130, 8, 2)])
def test_apply_update(ns, h, rows, cols, count):
    rng = np.random.default_rng(7 * rows + cols)
    W = rng.standard_normal((count, rows, cols), dtype=np.float32)
    m, n = min(rows, cols), max(rows, cols)
    Ow = o.bf16_rne_bits(rng.standard_normal((count, m, n), dtype=np.float32))
    lr, wd, sc = 0.02, 0.1, 1.7
    dW = dev(W)
    ns.muon_apply_update(h, rows, cols, count, dW, dev(Ow.view(np.int16)), lr, wd, sc)
    ns.muon_last_device_error(h)
    O = o.bf16_bits_to_f64(Ow)
    if rows > cols:                       # back to the weight's orientation
        O = np.swapaxes(O, -1, -2)
    ref = o.apply_update(W, O, lr, wd, sc)
    got = dW.cpu().numpy()
    bound = 1e-6 * (np.abs(W) + abs(lr * sc) * np.abs(O))
    assert (np.abs(got.astype(np.float64) - ref) <= bound).all()


# ----------------------------------------------------------------- step 3
NS_CASES = [
    (64, 128, 4, 5), (128, 128, 2, 5), (128, 256, 3, 5), (200, 328, 2, 5), (256, 1024, 2, 5),
    (384, 640, 3, 5), (8, 64, 2, 5), (64, 64, 1, 0), (64, 128, 2, 1), (128, 384, 2, 2),
    (512, 2048, 2, 5), (640, 1536, 2, 5), (136, 264, 1, 3), (1024, 1024, 1, 5),
]


@pytest.mark.parametrize("m,n,count,steps", NS_CASES)
def test_newton_schulz(ns, h, m, n, count, steps):
    rng = np.random.default_rng(m * 31 + n * 7 + count + steps)
    Xb = o.bf16_rne_bits(rng.standard_normal((count, m, n), dtype=np.float32))
    Xf = o.bf16_bits_to_f64(Xb)
    inv = np.array([1.0 / (np.linalg.norm(Xf[i]) + o.NORM_EPS) for i in range(count)],
                   dtype=np.float32)
    out = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    ns.muon_newton_schulz_bf16(h, m, n, count, dev(Xb.view(np.int16)), out, dev(inv), steps)
    ns.muon_last_device_error(h)
    got = o.bf16_bits_to_f64(u16(out))
    for i in range(count):
        ref = o.newton_schulz(Xf[i], 1.0 / float(inv[i]), steps)
        err = rel_fro(got[i], ref)
        assert err <= ns_tol(m, n), f"matrix {i}: rel err {err:.3e}"
        # Error model: the oracle's emulation rounds to BF16 exactly where
        # the kernels store (A, B', X), so the GPU's distance to the exact
        # iteration must match the emulation's up to accumulation order.
        # Any extra error of the kernels above ~1e-3 fails this.
        emu = o.newton_schulz(Xf[i], 1.0 / float(inv[i]), steps, emulate_bf16=True)
        model = rel_fro(emu, ref)
        assert err <= 1.15 * model + 5e-4, f"matrix {i}: {err:.3e} vs model {model:.3e}"


def test_newton_schulz_custom_coefficients(ns, h):
    m, n, count = 128, 256, 2
    co = (1.5, -0.5, 0.0)   # cubic iteration: a different polynomial
    rng = np.random.default_rng(3)
    Xb = o.bf16_rne_bits(rng.standard_normal((count, m, n), dtype=np.float32))
    Xf = o.bf16_bits_to_f64(Xb)
    inv = np.array([1.0 / (np.linalg.norm(Xf[i]) + o.NORM_EPS) for i in range(count)],
                   dtype=np.float32)
    out = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    ns.muon_newton_schulz_bf16(h, m, n, count, dev(Xb.view(np.int16)), out, dev(inv), 5, co)
    got = o.bf16_bits_to_f64(u16(out))
    for i in range(count):
        assert rel_fro(got[i], o.newton_schulz(Xf[i], 1.0 / float(inv[i]), 5, co)) <= NS_TOL


def test_newton_schulz_rejects_bad_shapes(ns, h):
    x = torch.zeros(64 * 128, dtype=torch.int16, device="cuda")
    inv = torch.ones(1, dtype=torch.float32, device="cuda")
    for m, n in [(128, 64), (60, 128), (64, 100)]:
        with pytest.raises(ns.MuonError) as ei:
            ns.muon_newton_schulz_bf16(h, m, n, 1, x, x.clone(), inv, 5)
        assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
    with pytest.raises(ns.MuonError):   # overlapping input and output
        ns.muon_newton_schulz_bf16(h, 64, 128, 1, x, x, inv, 5)


# ----------------------------------------------------------------- whole step
def run_step_and_check(ns, h, groups, arrays, lr=0.02, wd=0.1, mu=0.95, steps=5):
    """Run muon_step on device copies of arrays [(W, M, G, scale)] and check
    every matrix against the oracle."""
    dW = [dev(a[0]) for a in arrays]
    dM = [dev(a[1]) for a in arrays]
    dG = [dev(a[2]) for a in arrays]
    ns.muon_step(h, groups, dM, dG, dW, lr, wd, mu, steps)
    ns.muon_last_device_error(h)
    worst = 0.0
    for gi, (W, M, G, sc) in enumerate(arrays):
        Mg = dM[gi].cpu().numpy()
        Wg = dW[gi].cpu().numpy()
        for i in range(W.shape[0]):
            st = o.muon_step_matrix(W[i], M[i], G[i], lr=lr, wd=wd, mu=mu, ns_steps=steps,
                                    update_scale=sc)
            assert ulp_close(Mg[i], st.M_new).all()
            on = np.linalg.norm(st.O)
            dw = np.linalg.norm(Wg[i].astype(np.float64) - st.W_new.astype(np.float64))
            fp = 1e-6 * (np.linalg.norm(W[i]) + lr * abs(sc) * on)
            if on == 0.0:
                assert dw <= fp
                continue
            err = (dw - fp) / (lr * abs(sc) * on)
            worst = max(worst, err)
            tol = ns_tol(W.shape[1], W.shape[2])
            assert err <= tol, f"group {gi} matrix {i}: update error {err:.3e}"
    return worst


def test_step_tiny_workload(ns, h):
    from newton_schulz_03_gb300.workloads import WORKLOADS, make_group_numpy
    w = WORKLOADS["tiny"]
    groups, arrays = [], []
    for gi, g in enumerate(w.groups):
        W, M, G = make_group_numpy(w, gi)
        groups.append((g.rows, g.cols, g.count))
        arrays.append((W, M, G, 1.0))
    run_step_and_check(ns, h, groups, arrays, w.lr, w.wd, w.mu, w.ns_steps)


def test_step_mixed_ragged_groups(ns, h):
    rng = np.random.default_rng(77)
    shapes = [(128, 64, 3, 1.0), (64, 128, 2, 0.5), (37, 5, 2, 1.0), (100, 300, 1, 2.0),
              (300, 100, 2, 1.0), (64, 64, 0, 1.0), (1, 24, 2, 1.0), (264, 136, 1, 1.0)]
    groups, arrays = [], []
    for r, c, k, sc in shapes:
        groups.append((r, c, k, sc))
        arrays.append((rng.standard_normal((k, r, c), dtype=np.float32),
                       rng.standard_normal((k, r, c), dtype=np.float32),
                       rng.standard_normal((k, r, c), dtype=np.float32), sc))
    run_step_and_check(ns, h, groups, arrays)


def test_step_zero_matrix_only_decays(ns, h):
    rng = np.random.default_rng(5)
    W = rng.standard_normal((3, 96, 160), dtype=np.float32)
    Z = np.zeros_like(W)
    Z[1] = rng.standard_normal((96, 160), dtype=np.float32)   # matrix 1 is live
    dW, dM, dG = dev(W), dev(np.zeros_like(W)), dev(Z)
    ns.muon_step(h, [(96, 160, 3)], [dM], [dG], [dW], 0.02, 0.1, 0.95, 5)
    ns.muon_last_device_error(h)
    Wg = dW.cpu().numpy()
    decayed = o.apply_update(W, np.zeros_like(W), 0.02, 0.1)
    for i in (0, 2):
        assert ulp_close(Wg[i], decayed[i]).all()
    assert not ulp_close(Wg[1], decayed[1]).all()


def test_step_chunked_workspace(ns, ):
    """A workspace cap that holds two matrices forces several chunks; the
    result must not depend on chunking."""
    rng = np.random.default_rng(9)
    r, c, k = 256, 384, 5
    arrays = [(rng.standard_normal((k, r, c), dtype=np.float32),
               rng.standard_normal((k, r, c), dtype=np.float32),
               rng.standard_normal((k, r, c), dtype=np.float32), 1.0)]
    per = 2 * r * c * 2 + 2 * r * r * 2 + 64 * 4
    info = ns.muon_plan_describe([(r, c, k)], 5, 2 * per + 4096)
    assert info["n_chunks"] >= 3
    with ns.Handle(workspace_bytes_max=2 * per + 4096) as hh:
        run_step_and_check(ns, hh.value, [(r, c, k)], arrays)


@pytest.mark.parametrize("steps", [0, 1, 2, 4])
@pytest.mark.parametrize("r,c", [(384, 256), (96, 160)])
def test_step_iteration_counts(ns, h, steps, r, c):
    """muon_step with 0 (the normalised momentum), 1, 2 and 4 iterations: the
    final iterate lands in the buffer the apply kernel reads, on the
    CTA-pair path (m > 128) and the single-CTA path."""
    rng = np.random.default_rng(100 * steps + r)
    arrays = [tuple(rng.standard_normal((2, r, c), dtype=np.float32) for _ in range(3)) + (1.0,)]
    run_step_and_check(ns, h, [(r, c, 2)], arrays, steps=steps)


def test_step_host_buffers(ns, h):
    rng = np.random.default_rng(11)
    r, c, k = 192, 96, 3
    W, M, G = (rng.standard_normal((k, r, c), dtype=np.float32) for _ in range(3))
    Wh, Mh = torch.from_numpy(W.copy()).pin_memory(), torch.from_numpy(M.copy()).pin_memory()
    Gh = torch.from_numpy(G.copy()).pin_memory()
    ns.muon_step_host(h, [(r, c, k)], [Mh], [Gh], [Wh], 0.02, 0.1, 0.95, 5)
    for i in range(k):
        st = o.muon_step_matrix(W[i], M[i], G[i], lr=0.02, wd=0.1, mu=0.95)
        assert ulp_close(Mh.numpy()[i], st.M_new).all()
        err = np.linalg.norm(Wh.numpy()[i].astype(np.float64) - st.W_new) / (0.02 * np.linalg.norm(st.O))
        assert err <= NS_TOL + 1e-3


def test_invalid_arguments_launch_nothing(ns, h):
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    bad = [
        dict(groups=[(4, 4, 1)], M=[None], G=[x], W=[x]),
        dict(groups=[(4, 4, 1)], M=[x[1:]], G=[x], W=[x]),   # misaligned
        dict(groups=[(0, 4, 1)], M=[x], G=[x], W=[x]),
    ]
    before = ns.muon_kernel_stats(h)["total_launches"]
    for b in bad:
        with pytest.raises(ns.MuonError) as ei:
            ns.muon_step(h, b["groups"], b["M"], b["G"], b["W"], 0.02, 0.1, 0.95, 5)
        assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
    with pytest.raises(ns.MuonError):
        ns.muon_step(h, [(4, 4, 1)], [x], [x], [x], float("nan"), 0.1, 0.95, 5)
    assert ns.muon_kernel_stats(h)["total_launches"] == before


def test_nonfinite_norm_is_flagged(ns, h):
    M = np.zeros((1, 64, 64), dtype=np.float32)
    M[0, 3, 4] = np.inf
    dM, dG = dev(M), dev(np.zeros_like(M))
    X = torch.zeros((1, 64, 64), dtype=torch.int16, device="cuda")
    inv = torch.zeros(1, dtype=torch.float32, device="cuda")
    ns.muon_momentum_cast(h, 64, 64, 1, dM, dG, 0.9, X, inv)
    with pytest.raises(ns.MuonError) as ei:
        ns.muon_last_device_error(h)
    assert ei.value.status_name == "MUON_ERR_NONFINITE"
    ns.muon_last_device_error(h)   # the flag was cleared by the read


def test_kernel_timing_counts_launches(ns, h):
    rng = np.random.default_rng(1)
    W, M, G = (dev(rng.standard_normal((2, 128, 256), dtype=np.float32)) for _ in range(3))
    ns.muon_reset_kernel_stats(h)
    ns.muon_set_kernel_timing(h, True)
    ns.muon_step(h, [(128, 256, 2)], [M], [G], [W], 0.02, 0.1, 0.95, 5)
    st = ns.muon_kernel_stats(h)
    ns.muon_set_kernel_timing(h, False)
    assert st["launches"]["ns_gram"] == 5 and st["launches"]["ns_update"] == 5
    assert st["total_launches"] == 18
    assert all(v >= 0.0 for v in st["total_ms"].values())
    assert st["total_ms"]["ns_update"] > 0.0


def test_step_host_pipeline_matches_device_step(ns, h):
    """Host-buffer step over several pipeline pieces (>384 MB of state)
    equals the device-buffer step bit for bit, and sampled matrices match
    the oracle."""
    rng = np.random.default_rng(12)
    r, c, k = 1024, 1024, 40
    W, M, G = (rng.standard_normal((k, r, c), dtype=np.float32) * np.float32(0.05)
               for _ in range(3))
    Wh, Mh, Gh = (torch.from_numpy(a.copy()).pin_memory() for a in (W, M, G))
    ns.muon_step_host(h, [(r, c, k)], [Mh], [Gh], [Wh], 0.02, 0.1, 0.95, 5)
    dW, dM, dG = dev(W), dev(M), dev(G)
    ns.muon_step(h, [(r, c, k)], [dM], [dG], [dW], 0.02, 0.1, 0.95, 5)
    ns.muon_last_device_error(h)
    np.testing.assert_array_equal(Mh.numpy(), dM.cpu().numpy())
    np.testing.assert_array_equal(Wh.numpy(), dW.cpu().numpy())
    for i in (0, 39):
        st = o.muon_step_matrix(W[i], M[i], G[i], lr=0.02, wd=0.1, mu=0.95)
        err = np.linalg.norm(Wh.numpy()[i].astype(np.float64) - st.W_new) / (0.02 * np.linalg.norm(st.O))
        assert err <= NS_TOL + 1e-3


def test_step_host_mixed_groups_match_device_step(ns, h):
    """Host-buffer step over several groups (tall, wide, small) whose first
    and last pieces are split into ramps of growing and shrinking size
    equals the device-buffer step bit for bit."""
    rng = np.random.default_rng(13)
    groups = [(1024, 512, 40), (512, 1536, 30), (96, 160, 7)]
    host, devs = [], []
    for r, c, k in groups:
        W, M, G = (rng.standard_normal((k, r, c), dtype=np.float32) * np.float32(0.05)
                   for _ in range(3))
        host.append([torch.from_numpy(a.copy()).pin_memory() for a in (W, M, G)])
        devs.append([dev(a) for a in (W, M, G)])
    ns.muon_step_host(h, groups, [t[1] for t in host], [t[2] for t in host],
                      [t[0] for t in host], 0.02, 0.1, 0.95, 5)
    ns.muon_step(h, groups, [t[1] for t in devs], [t[2] for t in devs], [t[0] for t in devs],
                 0.02, 0.1, 0.95, 5)
    ns.muon_last_device_error(h)
    for hw, dw in zip(host, devs):
        np.testing.assert_array_equal(hw[0].numpy(), dw[0].cpu().numpy())
        np.testing.assert_array_equal(hw[1].numpy(), dw[1].cpu().numpy())


def test_bounded_wait_expires_and_context_survives(ns, h):
    """A device wait that can never complete gives up after its limit,
    reports MUON_ERR_TIMEOUT, and the context keeps working."""
    import time
    ns.muon_last_device_error(h)            # start clean
    t0 = time.perf_counter()
    ns.muon_selftest_bounded_wait(h, 50)
    with pytest.raises(ns.MuonError) as ei:
        ns.muon_last_device_error(h)
    waited = time.perf_counter() - t0
    assert ei.value.status_name == "MUON_ERR_TIMEOUT"
    assert 0.04 <= waited < 5.0
    ns.muon_last_device_error(h)            # cleared by the read
    # The GPU still computes correctly afterwards.
    m, n = 128, 256
    rng = np.random.default_rng(8)
    Xb = o.bf16_rne_bits(rng.standard_normal((1, m, n), dtype=np.float32))
    Xf = o.bf16_bits_to_f64(Xb)
    inv = np.array([1.0 / (np.linalg.norm(Xf[0]) + o.NORM_EPS)], dtype=np.float32)
    out = torch.zeros((1, m, n), dtype=torch.int16, device="cuda")
    ns.muon_newton_schulz_bf16(h, m, n, 1, dev(Xb.view(np.int16)), out, dev(inv), 5)
    ns.muon_last_device_error(h)
    got = o.bf16_bits_to_f64(u16(out))
    assert rel_fro(got[0], o.newton_schulz(Xf[0], 1.0 / float(inv[0]))) <= NS_TOL


def test_selftest_rejects_bad_limit(ns, h):
    for bad in (0, 2001):
        with pytest.raises(ns.MuonError) as ei:
            ns.muon_selftest_bounded_wait(h, bad)
        assert ei.value.status_name == "MUON_ERR_INVALID_ARG"


@pytest.mark.parametrize("rows,cols,count", [(256, 512, 2), (512, 256, 2), (200, 136, 1),
                                             (2048, 1536, 1)])
def test_step_equals_separate_entry_points(ns, h, rows, cols, count):
    """muon_step equals momentum_cast -> newton_schulz_bf16 ->
    apply_update called one after another, bit for bit (per-matrix results
    do not depend on how matrices are batched or padded)."""
    rng = np.random.default_rng(rows + cols)
    W, M, G = (rng.standard_normal((count, rows, cols), dtype=np.float32) for _ in range(3))
    lr, wd, mu = 0.02, 0.1, 0.95
    dW, dM, dG = dev(W), dev(M), dev(G)
    ns.muon_step(h, [(rows, cols, count)], [dM], [dG], [dW], lr, wd, mu, 5)
    m, n = min(rows, cols), max(rows, cols)
    sW, sM, sG = dev(W), dev(M), dev(G)
    X = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    O = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    inv = torch.zeros(count, dtype=torch.float32, device="cuda")
    ns.muon_momentum_cast(h, rows, cols, count, sM, sG, mu, X, inv)
    ns.muon_newton_schulz_bf16(h, m, n, count, X, O, inv, 5)
    ns.muon_apply_update(h, rows, cols, count, sW, O, lr, wd, 1.0)
    ns.muon_last_device_error(h)
    assert torch.equal(dM, sM)
    assert torch.equal(dW, sW)
