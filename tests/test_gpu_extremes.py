"""Extreme sizes through muon_step, checked against the CPU oracle:

* one matrix of more than 2^31 elements (65536 x 40000, tall, so it also
  runs through the transposing kernels) whose only non-zero entries form a
  small block near its far corner.  Zero padding is exact for the method
  (the norm, A = X X^T, the polynomial and the update all keep the zeros),
  so the step must leave every entry outside the block exactly zero and
  give the oracle's step of the block inside it.  Every flat offset of the
  block is above 2^31, so 32-bit index arithmetic anywhere shows up;
* the largest accepted dimension, 2^20, as the long side of wide and tall
  matrices (K = 2^20 in the Gram product), on both Newton-Schulz kernels;
* a group of more matrices than one elementwise launch covers (65535).
"""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import ulp_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

LR, WD, MU, STEPS = 0.02, 0.1, 0.95, 5


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


def update_error(Wg, st, W0):
    """Relative error of the applied update against the oracle's step."""
    on = np.linalg.norm(st.O)
    dw = np.linalg.norm(Wg.astype(np.float64) - st.W_new.astype(np.float64))
    fp = 1e-6 * (np.linalg.norm(W0) + LR * on)
    return (dw - fp) / (LR * on)


def test_single_matrix_beyond_int32_elements(ns, h):
    rows, cols = 65536, 40000                 # 2.62e9 elements; wide shape 40000 x 65536
    m, n = cols, rows
    need = 3 * rows * cols * 4 + 2 * m * n * 2 + 2 * m * m * 2 + (4 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on the device")
    kr, kc = 256, 384
    r0, c0 = rows - kr - 40, cols - kc - 8
    assert r0 * cols + c0 > 2**31 and c0 * rows + r0 > 2**31
    rng = np.random.default_rng(20240)
    Wb, Mb, Gb = (rng.standard_normal((kr, kc), dtype=np.float32) for _ in range(3))
    W = torch.zeros((1, rows, cols), dtype=torch.float32, device="cuda")
    M = torch.zeros_like(W)
    G = torch.zeros_like(W)
    for T, B in ((W, Wb), (M, Mb), (G, Gb)):
        T[0, r0:r0 + kr, c0:c0 + kc] = torch.from_numpy(B).cuda()
    ns.muon_step(h, [(rows, cols, 1)], [M], [G], [W], LR, WD, MU, STEPS)
    ns.muon_last_device_error(h)
    torch.cuda.synchronize()
    got = {}
    for name, T in (("W", W), ("M", M)):
        got[name] = T[0, r0:r0 + kr, c0:c0 + kc].cpu().numpy()
        T[0, r0:r0 + kr, c0:c0 + kc] = 0
        assert int(torch.count_nonzero(T)) == 0, f"{name}: non-zero entries outside the block"
    del W, M, G
    torch.cuda.empty_cache()
    st = o.muon_step_matrix(Wb, Mb, Gb, lr=LR, wd=WD, mu=MU, ns_steps=STEPS)
    assert ulp_close(got["M"], st.M_new).all()
    assert update_error(got["W"], st, Wb) <= 2e-2


@pytest.mark.parametrize("rows,cols,count", [(8, 1 << 20, 2), (1 << 20, 8, 1), (136, 1 << 20, 1)])
def test_largest_dimension(ns, h, rows, cols, count):
    rng = np.random.default_rng(rows + cols)
    W, M, G = (rng.standard_normal((count, rows, cols), dtype=np.float32) for _ in range(3))
    dW, dM, dG = (torch.from_numpy(a).cuda() for a in (W, M, G))
    ns.muon_step(h, [(rows, cols, count)], [dM], [dG], [dW], LR, WD, MU, STEPS)
    ns.muon_last_device_error(h)
    Mg, Wg = dM.cpu().numpy(), dW.cpu().numpy()
    del dW, dM, dG
    tol = 2e-2 if min(rows, cols) >= 64 else 4e-2
    for i in range(count):
        st = o.muon_step_matrix(W[i], M[i], G[i], lr=LR, wd=WD, mu=MU, ns_steps=STEPS)
        assert ulp_close(Mg[i], st.M_new).all()
        assert update_error(Wg[i], st, W[i]) <= tol


def test_more_matrices_than_one_launch(ns, h):
    rows, cols, count = 16, 8, 70000          # tall: a batch of 70000 wide 8 x 16 matrices
    rng = np.random.default_rng(65536)
    W, M, G = (rng.standard_normal((count, rows, cols), dtype=np.float32) for _ in range(3))
    dW, dM, dG = (torch.from_numpy(a).cuda() for a in (W, M, G))
    ns.muon_step(h, [(rows, cols, count)], [dM], [dG], [dW], LR, WD, MU, STEPS)
    ns.muon_last_device_error(h)
    Mg, Wg = dM.cpu().numpy(), dW.cpu().numpy()
    assert ulp_close(Mg, o.momentum_update(M, G, MU)).all()
    picks = sorted(set([0, 1, 65534, 65535, 65536, count - 1] +
                       list(rng.choice(count, 40, replace=False))))
    for i in picks:
        st = o.muon_step_matrix(W[i], M[i], G[i], lr=LR, wd=WD, mu=MU, ns_steps=STEPS)
        assert ulp_close(Mg[i], st.M_new).all()
        assert update_error(Wg[i], st, W[i]) <= 4e-2, f"matrix {i}"


@pytest.mark.parametrize("scale", [1e25, 1e15, 1e-25])
def test_extreme_momentum_scales(ns, h, scale):
    """The method is scale-invariant up to its 1e-7 in the norm.  At 1e25
    the FP32 partial sums of squares overflow (the norm is recomputed in
    FP64) and the norm (~6e27) is above 2^60, where the Gram product's FP32
    accumulator would overflow: the BF16 copy must come back scaled by a
    power of two with X * inv_norm unchanged, and the orthogonalised update
    must still match the oracle.  1e15 stays below both limits; at 1e-25
    the 1e-7 dominates the norm and the iteration is linear."""
    rows, cols, count = 384, 256, 2            # tall: runs as 256 x 384
    m, n = min(rows, cols), max(rows, cols)
    rng = np.random.default_rng(int(np.log10(scale)) + 100)
    M = (rng.standard_normal((count, rows, cols)) * scale).astype(np.float32)
    G = (rng.standard_normal((count, rows, cols)) * scale).astype(np.float32)
    dM, dG = torch.from_numpy(M.copy()).cuda(), torch.from_numpy(G).cuda()
    X = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    inv = torch.zeros(count, dtype=torch.float32, device="cuda")
    ns.muon_momentum_cast(h, rows, cols, count, dM, dG, MU, X, inv)
    O = torch.zeros_like(X)
    ns.muon_newton_schulz_bf16(h, m, n, count, X, O, inv, STEPS)
    ns.muon_last_device_error(h)
    Xg = o.bf16_bits_to_f64(X.cpu().numpy().view(np.uint16))
    Og = o.bf16_bits_to_f64(O.cpu().numpy().view(np.uint16))
    invg = inv.cpu().numpy().astype(np.float64)
    Mg = dM.cpu().numpy()
    for i in range(count):
        assert ulp_close(Mg[i], o.momentum_update(M[i], G[i], MU)).all()
        Mn = Mg[i]                               # the momentum the GPU cast
        Xw, _ = o.to_wide(o.bf16_rne(Mn))
        s = o.frobenius_scale(Mn)
        # the normalised input the products see (above ~1.8e19 per entry the
        # norm comes from the BF16 copy, within 2^-9 of the FP32 norm)
        rtol = 2e-6 if scale < 1e18 else 1e-3
        np.testing.assert_allclose(Xg[i] * invg[i], Xw / s, rtol=rtol, atol=0.0)
        ref = o.newton_schulz(Xw, s, STEPS)
        err = np.linalg.norm(Og[i] - ref) / np.linalg.norm(ref)
        assert err <= 2e-2, f"scale {scale:g} matrix {i}: {err:.3e}"
    if scale > 2.0**60:
        assert np.max(np.abs(Xg)) < 4.0      # the working copy was brought to unit scale


@pytest.mark.parametrize("m,n,rank", [(256, 384, 1), (256, 384, 5), (256, 384, 20),
                                      (256, 1024, 1), (256, 1024, 5), (512, 2048, 3)])
def test_rank_deficient_momentum(ns, h, m, n, rank):
    """A rank-r momentum: BF16 rounding of X puts noise in the null space,
    which the quintic amplifies (~a^5 = 480x), so even a BF16 emulation that
    rounds at exactly the GPU's points differs from the exact iteration by
    0.1-0.25 over the whole matrix -- a property of the format, not of the
    kernels.  What the method fixes is the output on the input's signal
    subspace, U_r^T O V_r, and the bound sigma(O) <= 1.2024 of the
    polynomial's band; both are checked against the oracle."""
    count = 2
    rng = np.random.default_rng(300 + rank + n)
    for i in range(count):
        M = (rng.standard_normal((m, rank)) @ rng.standard_normal((rank, n))).astype(np.float32)
        Xb = o.bf16_rne_bits(M)
        s = o.frobenius_scale(M)
        X = torch.from_numpy(Xb.view(np.int16).copy()).cuda().reshape(1, m, n)
        inv = torch.tensor([1.0 / s], dtype=torch.float32, device="cuda")
        O = torch.zeros_like(X)
        ns.muon_newton_schulz_bf16(h, m, n, 1, X, O, inv, STEPS)
        ns.muon_last_device_error(h)
        Og = o.bf16_bits_to_f64(O.cpu().numpy().view(np.uint16))[0]
        ref = o.newton_schulz(o.bf16_bits_to_f64(Xb), s, STEPS)
        U, _, Vt = np.linalg.svd(M.astype(np.float64), full_matrices=False)
        Ur, Vr = U[:, :rank], Vt[:rank].T
        pg, pr = Ur.T @ Og @ Vr, Ur.T @ ref @ Vr
        err = np.linalg.norm(pg - pr) / np.linalg.norm(pr)
        assert err <= 2e-2, f"rank {rank}: signal-subspace error {err:.3e}"
        assert np.linalg.svd(Og, compute_uv=False)[0] <= 1.2024 * (1 + 2.0**-7)


def test_low_rank_expert_in_a_batch(ns, h):
    """An MoE expert that received two tokens has a rank-2 gradient; with
    zero momentum its orthogonalised update must still have singular values
    inside the band and match the oracle on its signal subspace, next to
    full-rank experts of the same batch (which must match as usual)."""
    r, c, k = 512, 2048, 6
    rng = np.random.default_rng(2024)
    W = rng.standard_normal((k, r, c), dtype=np.float32)
    M = rng.standard_normal((k, r, c), dtype=np.float32) * np.float32(1e-3)
    G = rng.standard_normal((k, r, c), dtype=np.float32) * np.float32(1e-3)
    tok_in, tok_out = rng.standard_normal((r, 2)), rng.standard_normal((2, c))
    G[3] = (tok_in @ tok_out).astype(np.float32) * np.float32(1e-3)
    M[3] = 0.0
    dW, dM, dG = (torch.from_numpy(a.copy()).cuda() for a in (W, M, G))
    ns.muon_step(h, [(r, c, k)], [dM], [dG], [dW], LR, WD, MU, STEPS)
    ns.muon_last_device_error(h)
    Wg = dW.cpu().numpy()
    for i in range(k):
        st = o.muon_step_matrix(W[i], M[i], G[i], lr=LR, wd=WD, mu=MU, ns_steps=STEPS)
        if i != 3:
            assert update_error(Wg[i], st, W[i]) <= 2e-2
            continue
        # the kernel's decay, fmaf(-lr, wd, 1) rounded once to FP32
        decay = np.float64(np.float32(1.0 - np.float64(np.float32(LR)) * np.float64(np.float32(WD))))
        Og = (W[i].astype(np.float64) * decay - Wg[i].astype(np.float64)) / LR
        assert np.linalg.svd(Og, compute_uv=False)[0] <= 1.2024 * 1.01
        U, _, Vt = np.linalg.svd(G[i].astype(np.float64), full_matrices=False)
        Ur, Vr = U[:, :2], Vt[:2].T
        pg, pr = Ur.T @ Og @ Vr, Ur.T @ st.O @ Vr
        assert np.linalg.norm(pg - pr) / np.linalg.norm(pr) <= 2e-2
