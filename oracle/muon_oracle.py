"""CPU oracle for the one-GPU Muon step (test infrastructure only).

This module is the plain, slow, obviously-correct statement of what the
GPU path computes.  It is TEST INFRASTRUCTURE: only the test-suite, the
package smoke check and the CPU-baseline leg of the benchmark may import
it.  The product path never calls it and shares no code with it.

Sources (the pages describe the step in words only; no code is printed):

* [DN]   "Frontier Pre-training at Microsoft AI" (papercache deepnotes
         summary), Method details §5 "Scaling Muon to 16K GPUs", the
         five-step resharding pipeline.
* [XJ]   "Microsoft Reveals MAI-Base-2 Training Recipe" (xiaohu-jiedu,
         English), section "How to Make Parameter Updates Faster and More
         Stable?"; the same section on the Japanese page.
* [PT]   "MAI-Base-2 в 4–12 раз экономнее DeepSeek на предобучении"
         (promtime), section "Muon обошёл AdamW, но потребовал пересобирать
         матрицы между GPU".

What the pages fix: each data-parallel rank updates its FP32 momentum in
place and casts it to BF16 ([DN] step 1, [XJ]); same-shape matrices are
batched ([DN] step 2); every whole momentum matrix is orthogonalised by a
symmetry-aware Newton-Schulz operator ([DN] step 3, [XJ], [PT]); the
result is cast back to FP32 and applied to the weights ([DN] step 5).

What the pages leave open, and the reading taken here (each is also
listed in the design notes):

* Momentum: plain heavy-ball M <- mu*M + G (no Nesterov term).
* Newton-Schulz: the quintic iteration X <- aX + (bA + cA^2)X with
  A = X X^T, (a, b, c) = (3.4445, -4.7750, 2.0315), the same coefficients
  at every one of the (default 5) steps, on X0 = X / (||M'||_F + 1e-7).
  The Frobenius norm is taken of the FP32 momentum M' before the cast.
* A matrix with more rows than columns is orthogonalised as its
  transpose (so the Gram matrix is the smaller one) and transposed back.
* Weight update: decoupled decay W <- W(1 - lr*wd) - lr*s*O with a per
  group scale s (1 by default).
* The BF16 cast of the momentum is the method's own rounding point and is
  applied here; all later arithmetic is FP64 with no intermediate
  rounding unless ``emulate_bf16`` is requested (a diagnostic mode that
  rounds A, B and X to BF16 where the GPU stores them).

Parity pins: the iteration is pinned to the SVD closed form
X_N = U p^N(Sigma/s) V^T (p(x) = ax + bx^3 + cx^5), to orthogonal
equivariance, transpose and scale invariance and exact zero padding; the
BF16 cast to an independent library rounding; the momentum and weight
update to hand-computed special cases.  The end-to-end value has no
worked example on the pages: that single aspect is "parity unpinned" and
is covered by the pins above.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np

# Quintic Newton-Schulz coefficients and the normalisation epsilon of the
# tiny oracle-check configuration (the pages print neither).
NS_COEFFS: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315)
NS_STEPS: int = 5
NORM_EPS: float = 1e-7


# ---------------------------------------------------------------------------
# Scalars: the GPU receives hyper-parameters as FP32, so the oracle rounds
# them to FP32 first and then works in FP64.
# ---------------------------------------------------------------------------
def as_f32_scalar(x: float) -> float:
    """Value of ``x`` after rounding to IEEE binary32 (as a Python float)."""
    return float(np.float32(x))


# ---------------------------------------------------------------------------
# [DN] step 1, [XJ]: "cast to BF16".  Round-to-nearest-even from FP32.
# ---------------------------------------------------------------------------
def bf16_rne_bits(x32: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) of FP32 values, round to nearest even.

    BF16 keeps the upper 16 bits of the binary32 pattern.  The discarded
    low half decides the rounding: above 0x8000 rounds up, below rounds
    down, exactly 0x8000 rounds to the even upper half.  NaNs stay NaN
    (quiet bit forced); infinities and overflow behave as IEEE rounding.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    rounded = upper + round_up.astype(np.uint64)
    is_nan = np.isnan(x32)
    rounded = np.where(is_nan, upper | np.uint64(0x0040), rounded)
    return (rounded & np.uint64(0xFFFF)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of BF16 bit patterns, as float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def bf16_rne(x32: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 (RNE) -> exact float64 value."""
    return bf16_bits_to_f64(bf16_rne_bits(x32))


def _round_bf16_any(x: np.ndarray) -> np.ndarray:
    """Diagnostic: round an FP64 array to BF16 the way the GPU stores an
    FP32 accumulator (FP64 -> FP32 -> BF16)."""
    return bf16_rne(np.asarray(x, dtype=np.float64).astype(np.float32))


# ---------------------------------------------------------------------------
# [DN] step 1, [XJ], [PT]: update the FP32 momentum shard in place.
# ---------------------------------------------------------------------------
def momentum_update(M: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """M' = mu*M + G, evaluated in FP64 and stored back as FP32.

    Reading: plain heavy-ball momentum (the pages say only "update the
    momentum"); ``mu`` is taken at FP32 precision.
    """
    mu64 = as_f32_scalar(mu)
    out = mu64 * np.asarray(M, dtype=np.float64) + np.asarray(G, dtype=np.float64)
    return out.astype(np.float32)


# ---------------------------------------------------------------------------
# Orientation: a tall matrix (rows > cols) is orthogonalised as its
# transpose so that the Gram matrix X X^T is the smaller one.
# ---------------------------------------------------------------------------
def to_wide(X: np.ndarray) -> Tuple[np.ndarray, bool]:
    """Return (X or X^T, transposed?) so that the result has rows <= cols."""
    if X.shape[0] > X.shape[1]:
        return X.T, True
    return X, False


def frobenius_scale(M32: np.ndarray, eps: float = NORM_EPS) -> float:
    """s = ||M'||_F + eps, in FP64 (norm of the FP32 momentum)."""
    m = np.asarray(M32, dtype=np.float64)
    return float(np.sqrt(np.sum(m * m))) + eps


# ---------------------------------------------------------------------------
# [DN] step 3, [XJ], [PT]: Newton-Schulz orthogonalisation of a whole matrix.
# ---------------------------------------------------------------------------
def step_coeffs(coeffs, steps: int) -> List[Tuple[float, float, float]]:
    """Normalise ``coeffs`` to one (a, b, c) triple per step: a single
    triple is used at every step; a sequence of ``steps`` triples is a
    per-step schedule."""
    c = list(coeffs)
    if len(c) == 3 and not hasattr(c[0], "__len__"):
        return [tuple(float(v) for v in c)] * steps
    if len(c) != steps:
        raise ValueError("a coefficient schedule needs one (a, b, c) per step")
    return [tuple(float(v) for v in t) for t in c]


def newton_schulz(X: np.ndarray, s: float, steps: int = NS_STEPS,
                  coeffs: Sequence = NS_COEFFS,
                  emulate_bf16: bool = False) -> np.ndarray:
    """Quintic Newton-Schulz on a wide matrix X (rows <= cols).

    X0 = X / s; then ``steps`` times:  A = X X^T,  B = b A + c A A,
    X = a X + B X.  Plain FP64 matrix products, no symmetry shortcut.
    With ``emulate_bf16`` the products are rounded to BF16 where the GPU
    stores them: A, then B' = aI + bA + cA^2 (the linear term folded into
    the stored matrix), then each new X = B' X; the scale 1/s enters the
    first step as on the GPU.  That mode is a diagnostic, not the
    reference: both evaluation orders are the same polynomial.
    """
    X = np.asarray(X, dtype=np.float64)
    if X.shape[0] > X.shape[1]:
        raise ValueError("newton_schulz expects a wide matrix (rows <= cols)")
    sched = step_coeffs(coeffs, steps)
    if not emulate_bf16:
        Xk = X / s
        for a, b, c in sched:
            A = Xk @ Xk.T
            B = b * A + c * (A @ A)
            Xk = a * Xk + B @ Xk
        return Xk
    # Diagnostic path mirroring where the GPU rounds to BF16.
    Xk = X
    scale = 1.0 / s
    eye = np.eye(X.shape[0])
    for k, (a, b, c) in enumerate(sched):
        alpha = scale if k == 0 else 1.0
        A = _round_bf16_any((Xk @ Xk.T) * (alpha * alpha))
        B = _round_bf16_any(a * eye + b * A + c * (A @ A))
        Xk = _round_bf16_any(alpha * (B @ Xk))
    if steps == 0:
        Xk = _round_bf16_any(Xk * scale)
    return Xk


# ---------------------------------------------------------------------------
# [DN] step 5: cast the update back to FP32 and apply it to the weights.
# ---------------------------------------------------------------------------
def apply_update(W: np.ndarray, O: np.ndarray, lr: float, wd: float,
                 scale: float = 1.0) -> np.ndarray:
    """W' = W (1 - lr*wd) - lr*scale*O in FP64, stored as FP32.

    Reading: decoupled weight decay (the pages name decoupled decay in the
    hyper-parameter section and give no formula for the update itself).
    ``O`` has the weight's own orientation.
    """
    lr64, wd64, s64 = as_f32_scalar(lr), as_f32_scalar(wd), as_f32_scalar(scale)
    W64 = np.asarray(W, dtype=np.float64)
    O64 = np.asarray(O, dtype=np.float64)
    out = W64 * (1.0 - lr64 * wd64) - lr64 * s64 * O64
    return out.astype(np.float32)


# ---------------------------------------------------------------------------
# Method variants (not on the pages; common Muon variants, exposed as
# options).  Update scale rules multiply a group's own scale.
# ---------------------------------------------------------------------------
SCALE_NONE = 0          # 1
SCALE_SQRT_ASPECT = 1   # sqrt(max(1, rows / cols))   (rows = output dim)
SCALE_RMS_MATCH = 2     # rms_target * sqrt(max(rows, cols))


def update_scale_rule(rule: int, rows: int, cols: int, rms_target: float = 0.2) -> float:
    """Shape factor of the update for a weight of rows x cols, evaluated in
    FP32 as the library does (sqrt of an FP32 ratio / size)."""
    if rule == SCALE_NONE:
        return 1.0
    if rule == SCALE_SQRT_ASPECT:
        r = np.float32(max(1.0, np.float32(rows) / np.float32(cols)))
        return float(np.sqrt(r, dtype=np.float32))
    if rule == SCALE_RMS_MATCH:
        return float(np.float32(rms_target) * np.sqrt(np.float32(max(rows, cols)), dtype=np.float32))
    raise ValueError(f"unknown scale rule {rule}")


def nesterov_input(M_new: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Nesterov variant: the matrix orthogonalised is G + mu*M' (FP64 sum,
    stored as FP32), with M' the updated momentum."""
    mu64 = as_f32_scalar(mu)
    out = np.asarray(G, dtype=np.float64) + mu64 * np.asarray(M_new, dtype=np.float64)
    return out.astype(np.float32)


@dataclass
class MatrixStep:
    """Everything the oracle computes for one matrix."""
    M_new: np.ndarray      # FP32 momentum after the update (rows x cols)
    X_bf16: np.ndarray     # exact BF16 values of the cast, wide orientation
    transposed: bool       # True when the matrix was tall
    s: float               # ||M'||_F + eps
    O: np.ndarray          # Newton-Schulz output, weight orientation, FP64
    W_new: np.ndarray      # FP32 weights after the update


def muon_step_matrix(W: np.ndarray, M: np.ndarray, G: np.ndarray, *,
                     lr: float, wd: float, mu: float,
                     ns_steps: int = NS_STEPS,
                     coeffs: Sequence = NS_COEFFS,
                     eps: float = NORM_EPS, update_scale: float = 1.0,
                     emulate_bf16: bool = False, nesterov: bool = False) -> MatrixStep:
    """The whole step for one matrix, in the pages' order ([DN] steps 1-5,
    without the two all-to-all exchanges, which move data but do not
    change it).  With ``nesterov`` the orthogonalised matrix is G + mu*M'
    instead of M'."""
    M_new = momentum_update(M, G, mu)                      # step 1
    U = nesterov_input(M_new, G, mu) if nesterov else M_new
    Xb = bf16_rne(U)                                       # step 1: cast
    Xw, transposed = to_wide(Xb)
    s = frobenius_scale(U, eps)
    Ow = newton_schulz(Xw, s, ns_steps, coeffs, emulate_bf16)   # step 3
    O = Ow.T if transposed else Ow
    W_new = apply_update(W, O, lr, wd, update_scale)       # step 5
    return MatrixStep(M_new=M_new, X_bf16=Xw, transposed=transposed, s=s,
                      O=O, W_new=W_new)


def group_by_wide_shape(shapes: Sequence[Tuple[int, int]]) -> List[Tuple[Tuple[int, int], List[int]]]:
    """[DN] step 2: batch parameters of identical shape.  Matrices are keyed
    by their wide shape (min, max), so a tall matrix joins the batch of its
    transpose.  Returns [(wide_shape, [indices in input order])] in order
    of first appearance."""
    order: List[Tuple[int, int]] = []
    members = {}
    for i, (r, c) in enumerate(shapes):
        key = (min(r, c), max(r, c))
        if key not in members:
            members[key] = []
            order.append(key)
        members[key].append(i)
    return [(k, members[k]) for k in order]


def muon_step(weights: Sequence[np.ndarray], momenta: Sequence[np.ndarray],
              grads: Sequence[np.ndarray], *, lr: float, wd: float, mu: float,
              ns_steps: int = NS_STEPS, coeffs: Sequence[float] = NS_COEFFS,
              eps: float = NORM_EPS, update_scales: Sequence[float] | None = None
              ) -> List[MatrixStep]:
    """Muon step over a list of matrices, one matrix at a time (grouping
    changes the schedule, not the result)."""
    out = []
    for i, (W, M, G) in enumerate(zip(weights, momenta, grads)):
        sc = 1.0 if update_scales is None else update_scales[i]
        out.append(muon_step_matrix(W, M, G, lr=lr, wd=wd, mu=mu,
                                    ns_steps=ns_steps, coeffs=coeffs,
                                    eps=eps, update_scale=sc))
    return out


# ---------------------------------------------------------------------------
# Work model used by the benchmark's FLOP accounting.
# ---------------------------------------------------------------------------
def ns_algorithmic_flops(m: int, n: int, steps: int = NS_STEPS) -> int:
    """Flops the symmetric method executes per matrix (m <= n): per step
    the Gram product m^2 n (half of 2 m^2 n), the symmetric square m^3 and
    the update product 2 m^2 n."""
    return steps * (3 * m * m * n + m * m * m)


def ns_dense_flops(m: int, n: int, steps: int = NS_STEPS) -> int:
    """Dense-equivalent flops per matrix (no symmetry): 5*(4 m^2 n + 2 m^3)."""
    return steps * (4 * m * m * n + 2 * m * m * m)


# ---------------------------------------------------------------------------
# AdamW companion for the parameters Muon does not handle (embeddings,
# norms, scalars): "Microsoft Reveals MAI-Base-2 Training Recipe", section
# "How to Make Parameter Updates Faster and More Stable?" (Muon for 2-D
# non-embedding matrices, AdamW for the rest).  The pages give no formula;
# this is the standard decoupled-decay AdamW with bias correction.
# ---------------------------------------------------------------------------
def adamw_step(p: np.ndarray, g: np.ndarray, m: np.ndarray, v: np.ndarray, *,
               lr: float, beta1: float, beta2: float, eps: float, wd: float,
               step: int):
    """One AdamW step (step >= 1) in FP64 on FP32 inputs; returns the new
    (p, m, v) as FP32.  p <- p (1 - lr wd); m <- b1 m + (1 - b1) g;
    v <- b2 v + (1 - b2) g^2; p <- p - lr m_hat / (sqrt(v_hat) + eps) with
    m_hat = m / (1 - b1^t), v_hat = v / (1 - b2^t)."""
    lr, b1, b2 = as_f32_scalar(lr), as_f32_scalar(beta1), as_f32_scalar(beta2)
    eps, wd = as_f32_scalar(eps), as_f32_scalar(wd)
    p64 = np.asarray(p, np.float64) * (1.0 - lr * wd)
    g64 = np.asarray(g, np.float64)
    m64 = b1 * np.asarray(m, np.float64) + (1.0 - b1) * g64
    v64 = b2 * np.asarray(v, np.float64) + (1.0 - b2) * g64 * g64
    m_hat = m64 / (1.0 - b1 ** step)
    v_hat = v64 / (1.0 - b2 ** step)
    p64 = p64 - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p64.astype(np.float32), m64.astype(np.float32), v64.astype(np.float32)
