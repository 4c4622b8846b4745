"""Pins for the CPU oracle, each against something other than the oracle.

* BF16 cast: bit-for-bit against PyTorch's CPU float32->bfloat16
  conversion (an independent round-to-nearest-even) and hand-worked ties.
* Newton-Schulz: the SVD closed form X_N = U p^N(Sigma/s) V^T, with the
  scalar map p(x) = a x + b x^3 + c x^5 iterated here on plain floats; the
  singular-value band that map produces; orthogonal equivariance,
  transpose, scale invariance, zero input and exact zero padding.
* Momentum and weight update: hand-computed special cases in exact
  rational arithmetic on the FP32 scalars.
* Mutation check: deliberately wrong variants of the iteration (planted
  here, on the CPU) must fail the closed-form pin.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import muon_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def p_iter(x, steps=o.NS_STEPS, coeffs=o.NS_COEFFS):
    a, b, c = coeffs
    y = np.array(x, dtype=np.float64)
    for _ in range(steps):
        y = a * y + b * y ** 3 + c * y ** 5
    return y


def closed_form(X, s, steps=o.NS_STEPS, coeffs=o.NS_COEFFS):
    U, S, Vt = np.linalg.svd(X / s, full_matrices=False)
    return (U * p_iter(S, steps, coeffs)) @ Vt


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------
# Configuration fixture
# --------------------------------------------------------------------------
def test_defaults_match_configuration_fixture():
    with open(os.path.join(GOLDEN, "ns_configuration.json")) as f:
        cfg = json.load(f)
    assert tuple(cfg["coeffs"]) == o.NS_COEFFS
    assert cfg["steps"] == o.NS_STEPS
    assert cfg["eps"] == o.NORM_EPS


# --------------------------------------------------------------------------
# BF16 round-to-nearest-even
# --------------------------------------------------------------------------
def _torch_bits(x32):
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_matches_library_rounding_random():
    rng = np.random.default_rng(11)
    # Every exponent range: subnormals to near overflow, both signs.
    mant = rng.uniform(1.0, 2.0, 200000)
    expo = rng.integers(-140, 127, 200000)
    sign = rng.choice([-1.0, 1.0], 200000)
    x = (sign * mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    np.testing.assert_array_equal(o.bf16_rne_bits(x), _torch_bits(x))


def test_bf16_matches_library_rounding_ties():
    rng = np.random.default_rng(12)
    # Bit patterns whose low half is exactly 0x8000 (ties), 0x7FFF, 0x8001.
    hi = rng.integers(0, 0x7F7F, 50000, dtype=np.uint32)
    for low in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
        u = (hi << np.uint32(16)) | np.uint32(low)
        x = u.view(np.float32)
        np.testing.assert_array_equal(o.bf16_rne_bits(x), _torch_bits(x))


def test_bf16_hand_cases():
    one_tie = np.float32(1.0 + 2.0 ** -8)            # halfway 1 | 1+2^-7 -> even (1)
    odd_tie = np.float32(1.0 + 3 * 2.0 ** -8)        # halfway 1+2^-7 | 1+2^-6 -> 1+2^-6
    above = np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)  # just above halfway -> up
    vals = o.bf16_rne(np.array([one_tie, odd_tie, above, -odd_tie], dtype=np.float32))
    assert list(vals) == [1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -(1.0 + 2.0 ** -6)]
    big = np.array([np.finfo(np.float32).max, np.inf, -np.inf], dtype=np.float32)
    assert list(o.bf16_rne(big)) == [np.inf, np.inf, -np.inf]
    assert np.isnan(o.bf16_rne(np.array([np.nan], dtype=np.float32))[0])
    assert o.bf16_rne_bits(np.array([0.0, -0.0], dtype=np.float32)).tolist() == [0, 0x8000]


# --------------------------------------------------------------------------
# Newton-Schulz against the SVD closed form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("m,n,rank", [(4, 4, 4), (5, 9, 5), (16, 40, 16), (12, 30, 5),
                                      (32, 32, 31), (1, 7, 1), (64, 128, 64)])
def test_ns_closed_form(m, n, rank):
    rng = np.random.default_rng(100 + m * 7 + n + rank)
    X = rng.standard_normal((m, rank)) @ rng.standard_normal((rank, n))
    s = np.linalg.norm(X) + o.NORM_EPS
    got = o.newton_schulz(X, s)
    want = closed_form(X, s)
    assert rel(got, want) < 1e-10


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 7])
def test_ns_closed_form_steps(steps):
    rng = np.random.default_rng(5 + steps)
    X = rng.standard_normal((10, 24))
    s = np.linalg.norm(X) + o.NORM_EPS
    assert rel(o.newton_schulz(X, s, steps), closed_form(X, s, steps)) < 1e-10


def test_ns_closed_form_other_coefficients():
    rng = np.random.default_rng(9)
    X = rng.standard_normal((8, 20))
    s = np.linalg.norm(X) + o.NORM_EPS
    co = (1.5, -0.5, 0.0)   # cubic Newton-Schulz
    assert rel(o.newton_schulz(X, s, 5, co), closed_form(X, s, 5, co)) < 1e-10


def test_ns_band_of_scalar_map():
    x = np.logspace(np.log10(3e-3), 0.0, 100001)
    y = p_iter(x)
    assert abs(y.min() - 0.6818) < 1e-4 and abs(y.max() - 1.2024) < 1e-4
    x2 = np.logspace(-2, 0.0, 100001)
    assert abs(p_iter(x2).max() - 1.1344) < 1e-4


def test_ns_output_shares_singular_vectors_with_polar_factor():
    rng = np.random.default_rng(21)
    U, _ = np.linalg.qr(rng.standard_normal((24, 24)))
    V, _ = np.linalg.qr(rng.standard_normal((60, 24)))
    sig = np.logspace(0, -2, 24)            # normalised sigma spans 1 .. 1e-2
    X = (U * sig) @ V.T
    s = np.linalg.norm(X) + o.NORM_EPS
    O = o.newton_schulz(X, s)
    polar = U @ V.T
    # O = U diag(d) V^T with d in the band: U^T O V is diagonal.
    D = U.T @ O @ V
    assert np.abs(D - np.diag(np.diag(D))).max() < 1e-10
    d = np.diag(D)
    sn = sig / s
    assert np.all(d[sn >= 3e-3] >= 0.6818 - 1e-9) and np.all(d[sn >= 3e-3] <= 1.2024 + 1e-9)
    # ...and the same singular vectors as the polar factor U V^T.
    assert np.abs(U.T @ polar @ V - np.eye(24)).max() < 1e-12


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------
def test_ns_orthogonal_equivariance():
    rng = np.random.default_rng(31)
    X = rng.standard_normal((12, 28))
    Q, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    P, _ = np.linalg.qr(rng.standard_normal((28, 28)))
    s = np.linalg.norm(X) + o.NORM_EPS
    lhs = o.newton_schulz(Q @ X @ P, s)
    rhs = Q @ o.newton_schulz(X, s) @ P
    assert rel(lhs, rhs) < 1e-10


def test_step_transpose_invariance():
    rng = np.random.default_rng(32)
    W, M, G = (rng.standard_normal((20, 9)).astype(np.float32) for _ in range(3))
    kw = dict(lr=0.02, wd=0.1, mu=0.95)
    tall = o.muon_step_matrix(W, M, G, **kw)
    wide = o.muon_step_matrix(W.T.copy(), M.T.copy(), G.T.copy(), **kw)
    assert tall.transposed and not wide.transposed
    assert tall.O.shape == (20, 9) and wide.O.shape == (9, 20)
    assert rel(tall.O, wide.O.T) < 1e-12
    np.testing.assert_array_equal(tall.W_new, wide.W_new.T)


def test_ns_scale_invariance():
    rng = np.random.default_rng(33)
    X = rng.standard_normal((6, 15))
    for alpha in (1e-3, 7.0):
        # With eps = 0 the normalisation removes the scale exactly.
        a = o.newton_schulz(alpha * X, alpha * np.linalg.norm(X))
        b = o.newton_schulz(X, np.linalg.norm(X))
        assert rel(a, b) < 1e-12


def test_ns_zero_input_is_zero():
    X = np.zeros((8, 16))
    s = o.frobenius_scale(X.astype(np.float32))
    assert s == o.NORM_EPS
    assert np.all(o.newton_schulz(X, s) == 0.0)


@pytest.mark.parametrize("pad_rows,pad_cols", [(0, 5), (3, 0), (4, 9)])
def test_ns_zero_padding_exact(pad_rows, pad_cols):
    rng = np.random.default_rng(34)
    X = rng.standard_normal((10, 22))
    s = np.linalg.norm(X) + o.NORM_EPS
    Xp = np.zeros((10 + pad_rows, 22 + pad_cols))
    Xp[:10, :22] = X
    Op = o.newton_schulz(Xp, s)
    assert np.all(Op[10:, :] == 0.0) and np.all(Op[:, 22:] == 0.0)
    assert rel(Op[:10, :22], o.newton_schulz(X, s)) < 1e-13


# --------------------------------------------------------------------------
# Momentum and weight update: exact rational arithmetic on FP32 scalars
# --------------------------------------------------------------------------
def _f32_exact(x):
    return Fraction(float(np.float32(x)))


def test_momentum_hand_cases():
    M = np.array([1.0, 2.0, -3.0, 0.25], dtype=np.float32)
    G = np.array([0.5, -1.0, 1.5, 0.0], dtype=np.float32)
    out = o.momentum_update(M, G, 0.5)
    assert out.tolist() == [1.0, 0.0, 0.0, 0.125]
    np.testing.assert_array_equal(o.momentum_update(M, G, 0.0), G)
    mu = _f32_exact(0.95)
    want = [np.float32(float(mu * Fraction(float(m)) + Fraction(float(g))))
            for m, g in zip(M, G)]
    np.testing.assert_array_equal(o.momentum_update(M, G, 0.95), np.array(want))


def test_apply_update_hand_cases():
    W = np.array([1.0, -2.0, 0.0], dtype=np.float32)
    O = np.array([1.0, 0.5, -1.0])
    lr, wd = _f32_exact(0.5), _f32_exact(0.1)
    want = [np.float32(float(Fraction(float(w)) * (1 - lr * wd) - lr * Fraction(float(x))))
            for w, x in zip(W, O)]
    np.testing.assert_array_equal(o.apply_update(W, O, 0.5, 0.1), np.array(want))
    # scale multiplies the update only
    got = o.apply_update(W, O, 0.5, 0.0, scale=2.0)
    np.testing.assert_array_equal(got, np.array([0.0, -2.5, 1.0], dtype=np.float32))


def test_step_zero_momentum_and_grad_only_decays():
    rng = np.random.default_rng(35)
    W = rng.standard_normal((6, 10)).astype(np.float32)
    Z = np.zeros_like(W)
    st = o.muon_step_matrix(W, Z, Z, lr=0.02, wd=0.1, mu=0.95)
    assert np.all(st.M_new == 0.0) and np.all(st.O == 0.0)
    np.testing.assert_array_equal(st.W_new, o.apply_update(W, np.zeros_like(W), 0.02, 0.1))


def test_step_mu_zero_is_gradient():
    rng = np.random.default_rng(36)
    W, M, G = (rng.standard_normal((8, 8)).astype(np.float32) for _ in range(3))
    st = o.muon_step_matrix(W, M, G, lr=0.02, wd=0.1, mu=0.0)
    np.testing.assert_array_equal(st.M_new, G)
    s = np.linalg.norm(G.astype(np.float64)) + o.NORM_EPS
    assert abs(st.s - s) < 1e-12 * s
    assert rel(st.O, closed_form(o.bf16_rne(G), s)) < 1e-10


def test_step_ns_steps_zero_is_normalised_momentum():
    rng = np.random.default_rng(37)
    W, M, G = (rng.standard_normal((5, 7)).astype(np.float32) for _ in range(3))
    st = o.muon_step_matrix(W, M, G, lr=0.02, wd=0.1, mu=0.9, ns_steps=0)
    assert rel(st.O, o.bf16_rne(st.M_new) / st.s) < 1e-15


# --------------------------------------------------------------------------
# Grouping and flop model
# --------------------------------------------------------------------------
def test_group_by_wide_shape():
    groups = o.group_by_wide_shape([(1536, 4096), (4096, 1536), (64, 64), (4096, 1536)])
    assert groups == [((1536, 4096), [0, 1, 3]), ((64, 64), [2])]


def test_flop_model():
    assert o.ns_algorithmic_flops(2, 3, 1) == 3 * 4 * 3 + 8
    assert o.ns_dense_flops(2, 3, 1) == 4 * 4 * 3 + 2 * 8


# --------------------------------------------------------------------------
# Mutation check: wrong iterations must fail the closed-form pin
# --------------------------------------------------------------------------
def _mutant(kind):
    def ns(X, s, steps=o.NS_STEPS, coeffs=o.NS_COEFFS):
        a, b, c = coeffs
        Xk = X / s
        for _ in range(steps):
            A = Xk @ Xk.T
            if kind == "drop_cubic":
                B = c * (A @ A)
            elif kind == "sign_c":
                B = b * A - c * (A @ A)
            elif kind == "swap_bc":
                B = c * A + b * (A @ A)
            elif kind == "right_multiply":
                B = b * A + c * (A @ A)
                Xk = a * Xk + Xk @ B
                continue
            elif kind == "no_normalise":
                if Xk is not None and _ == 0:
                    Xk = Xk * s
                B = b * A + c * (A @ A)
            elif kind == "gram_transposed":
                At = Xk.T @ Xk
                Xk = a * Xk + Xk @ (b * At + c * (At @ At))
                continue
            else:
                B = b * A + c * (A @ A)
            Xk = a * Xk + B @ Xk
        return Xk
    return ns


@pytest.mark.parametrize("kind", ["drop_cubic", "sign_c", "swap_bc", "right_multiply",
                                  "no_normalise"])
def test_closed_form_rejects_mutants(kind):
    rng = np.random.default_rng(41)
    # Square, so that multiplying B on the wrong side is a valid product
    # that gives a different (wrong) answer.
    X = rng.standard_normal((6, 6)) @ np.diag(np.linspace(0.2, 3.0, 6)) @ rng.standard_normal((6, 6))
    s = np.linalg.norm(X) + o.NORM_EPS
    assert rel(_mutant("none")(X, s), closed_form(X, s)) < 1e-10
    with np.errstate(all="ignore"):
        r = rel(_mutant(kind)(X, s), closed_form(X, s))
    assert not (r < 1e-3)   # NaN (divergence) counts as a rejection


def test_closed_form_does_not_distinguish_gram_side():
    # X (X^T X) == (X X^T) X exactly in theory, so the side of the Gram
    # product is a schedule choice, not a correctness one.
    rng = np.random.default_rng(42)
    X = rng.standard_normal((5, 11))
    s = np.linalg.norm(X) + o.NORM_EPS
    assert rel(_mutant("gram_transposed")(X, s), closed_form(X, s)) < 1e-10


def test_emulated_bf16_mode_is_close_to_exact():
    # The diagnostic mode rounds where the GPU stores products; its error
    # against the exact iteration is the BF16 floor the GPU tests allow for.
    rng = np.random.default_rng(50)
    X = o.bf16_rne(rng.standard_normal((64, 128)).astype(np.float32))
    s = np.linalg.norm(X) + o.NORM_EPS
    err = rel(o.newton_schulz(X, s, emulate_bf16=True), o.newton_schulz(X, s))
    assert 1e-4 < err < 2e-2


def test_error_model_check_detects_rounding_mistakes():
    # The GPU parity tests require the kernels' error against the exact
    # iteration to match the emulation's (rounding where the kernels store)
    # within 15% + 5e-4.  Mistakes planted here, in a copy of the emulated
    # iteration on the CPU -- one extra BF16 rounding of c A^2, or rounding
    # before the a I term is added -- stay under the plain 2e-2 bar but
    # fail that check.
    rng = np.random.default_rng(52)
    X = o.bf16_rne(rng.standard_normal((128, 256)).astype(np.float32))
    s = np.linalg.norm(X) + o.NORM_EPS
    ref = o.newton_schulz(X, s)
    model = rel(o.newton_schulz(X, s, emulate_bf16=True), ref)
    rnd = o._round_bf16_any
    a, b, c = o.NS_COEFFS

    def planted(kind):
        Y = X / s
        for _ in range(5):
            A = rnd(Y @ Y.T)
            eye = np.eye(A.shape[0])
            if kind == "extra_round":
                B = rnd(b * A + rnd(c * (A @ A)) + a * eye)
            else:
                B = rnd(rnd(b * A + c * (A @ A)) + a * eye)
            Y = rnd(B @ Y)
        return Y

    for kind in ("extra_round", "early_round"):
        err = rel(planted(kind), ref)
        assert err <= 2e-2 and err > 1.15 * model + 5e-4, (kind, err, model)


def test_emulated_bf16_floor_on_rank_deficient_input():
    # Rank-1 input: BF16 rounding puts noise in the null space that the
    # quintic amplifies, so the emulation (rounding where the GPU stores)
    # differs from the exact iteration far beyond 2e-2 over the whole
    # matrix, while on the input's signal subspace the two agree closely.
    # This is the floor behind the rank-deficient tolerance of the GPU tests.
    rng = np.random.default_rng(51)
    M = np.outer(rng.standard_normal(128), rng.standard_normal(192)).astype(np.float32)
    X = o.bf16_rne(M)
    s = o.frobenius_scale(M)
    emu, ex = o.newton_schulz(X, s, emulate_bf16=True), o.newton_schulz(X, s)
    assert rel(emu, ex) > 5e-2
    U, _, Vt = np.linalg.svd(M.astype(np.float64), full_matrices=False)
    u, v = U[:, :1], Vt[:1].T
    assert rel(u.T @ emu @ v, u.T @ ex @ v) < 5e-3
    assert np.linalg.svd(emu, compute_uv=False)[0] <= 1.2024


# --------------------------------------------------------------------------
# Method variants
# --------------------------------------------------------------------------
def test_coefficient_schedule_closed_form():
    rng = np.random.default_rng(60)
    X = rng.standard_normal((9, 21))
    s = np.linalg.norm(X) + o.NORM_EPS
    sched = [(4.0, -5.0, 2.0), (3.4445, -4.7750, 2.0315), (2.5, -2.0, 0.6), (1.5, -0.5, 0.0)]
    U, S, Vt = np.linalg.svd(X / s, full_matrices=False)
    y = S.copy()
    for a, b, c in sched:
        y = a * y + b * y ** 3 + c * y ** 5
    assert rel(o.newton_schulz(X, s, 4, sched), (U * y) @ Vt) < 1e-10
    # A constant schedule equals the single-triple form.
    const = [o.NS_COEFFS] * 5
    assert rel(o.newton_schulz(X, s, 5, const), o.newton_schulz(X, s)) == 0.0
    with pytest.raises(ValueError):
        o.newton_schulz(X, s, 3, sched)


def test_nesterov_hand_case():
    M = np.array([[1.0, 2.0]], dtype=np.float32)
    G = np.array([[0.5, -1.0]], dtype=np.float32)
    M_new = o.momentum_update(M, G, 0.5)          # [1.0, 0.0]
    assert o.nesterov_input(M_new, G, 0.5).tolist() == [[1.0, -1.0]]
    # mu = 0: Nesterov and heavy ball both orthogonalise G.
    rng = np.random.default_rng(61)
    W, M, G = (rng.standard_normal((6, 10)).astype(np.float32) for _ in range(3))
    a = o.muon_step_matrix(W, M, G, lr=0.02, wd=0.1, mu=0.0, nesterov=True)
    b = o.muon_step_matrix(W, M, G, lr=0.02, wd=0.1, mu=0.0, nesterov=False)
    np.testing.assert_array_equal(a.W_new, b.W_new)


def test_nesterov_orthogonalises_g_plus_mu_m():
    rng = np.random.default_rng(62)
    W, M, G = (rng.standard_normal((8, 12)).astype(np.float32) for _ in range(3))
    st = o.muon_step_matrix(W, M, G, lr=0.02, wd=0.1, mu=0.9, nesterov=True)
    U = (G.astype(np.float64) + np.float64(np.float32(0.9)) * st.M_new.astype(np.float64)).astype(np.float32)
    s = np.linalg.norm(U.astype(np.float64)) + o.NORM_EPS
    assert rel(st.O, closed_form(o.bf16_rne(U), s)) < 1e-10


@pytest.mark.parametrize("rows,cols,rule,want", [
    (4096, 1536, o.SCALE_SQRT_ASPECT, np.sqrt(4096 / 1536)), (1536, 4096, o.SCALE_SQRT_ASPECT, 1.0),
    (64, 64, o.SCALE_SQRT_ASPECT, 1.0), (1536, 4096, o.SCALE_RMS_MATCH, 0.2 * 64.0),
    (100, 36, o.SCALE_RMS_MATCH, 0.2 * 10.0), (7, 5, o.SCALE_NONE, 1.0)])
def test_update_scale_rules(rows, cols, rule, want):
    assert abs(o.update_scale_rule(rule, rows, cols) - want) <= 1e-6 * want


# --------------------------------------------------------------------------
# AdamW companion
# --------------------------------------------------------------------------
def test_adamw_matches_torch_reference():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(70)
    p0 = rng.standard_normal(1000).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    tp = torch.nn.Parameter(torch.from_numpy(p0.astype(np.float64)))
    f32 = o.as_f32_scalar
    opt = torch.optim.AdamW([tp], lr=f32(hp["lr"]), betas=(f32(hp["beta1"]), f32(hp["beta2"])),
                            eps=f32(hp["eps"]), weight_decay=f32(hp["wd"]), foreach=False)
    for t in range(1, 6):
        g = rng.standard_normal(1000).astype(np.float32)
        p, m, v = o.adamw_step(p, g, m, v, step=t, **hp)
        # The torch reference runs in FP64 on the same FP32 inputs each step.
        tp.data = torch.from_numpy(p_prev.astype(np.float64)) if t > 1 else tp.data
        tp.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        p_prev = p
        np.testing.assert_allclose(tp.data.numpy(), p.astype(np.float64), rtol=2e-7, atol=1e-9)


def test_adamw_first_step_is_signed_lr():
    # At t = 1 with zero state: m_hat = g, v_hat = g^2, so the update is
    # lr * g / (|g| + eps) -- the sign of g times lr, minus decay.
    g = np.array([2.0, -0.5, 1e-3], dtype=np.float32)
    p = np.array([1.0, 1.0, 1.0], dtype=np.float32)
    z = np.zeros(3, dtype=np.float32)
    p1, m1, v1 = o.adamw_step(p, g, z, z, lr=0.01, beta1=0.9, beta2=0.99, eps=1e-12, wd=0.0,
                              step=1)
    np.testing.assert_allclose(p1, [0.99, 1.01, 0.99], rtol=1e-6)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-6)
    np.testing.assert_allclose(v1, 0.01 * g * g, rtol=1e-5)
