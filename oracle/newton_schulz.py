"""Newton-Schulz orthogonalisation, oracle version (test infrastructure).

The pages ("Support Muon in BF16_Optimizer with FP32 gradient accumulation",
validation table; "Run Muon once per optimizer step under ZeRO-3, not once
per micro-batch", review thread) name two methods, "standard" and "gram",
with "gram" the default, and give no formula.  Readings used here:

* Quintic map f(x) = a x + b x^3 + c x^5 with (a, b, c) =
  (3.4445, -4.7750, 2.0315), applied 5 times by default: the usual Muon
  coefficients, stated as an assumption.
* Normalisation: X0 = G / (||G||_F + 1e-7).  A zero matrix gives zero.
* Orientation: a matrix with rows > cols is transposed first, iterated as
  X (m x n, m <= n) and transposed back; rows == cols is not transposed.
* standard: per step  A = X X^T,  B = b A + c A A,  X <- a X + B X.
* gram: the same polynomial map run on the Gram matrix.  With
  R = X0 X0^T and Q = I, each step forms P = a I + b R + c R R, then
  Q <- P Q and (except after the last step) R <- (P R) P; finally
  Y = Q X0.  Because P is a polynomial in R, X_k = Q_k X0 and
  R_k = X_k X_k^T hold in exact arithmetic, so gram equals standard.

Two arithmetic modes:

* ``"exact"``: everything in float64.
* ``"bf16"``: emulates BF16 operands with FP32 accumulation.  The normalised
  X0 is rounded to bfloat16; each matrix product is accumulated in float64,
  rounded to float32, combined with its addend in float32 as
  ``alpha*acc + beta*E (+ gamma on the diagonal)`` and the result rounded to
  bfloat16.  standard: A, B and X are rounded this way every step.
  gram: only the m x n products use BF16 operands -- R0 = X0 X0^T is kept in
  float32 (its inputs are bfloat16), the m x m recurrence (P, Q, P R, R)
  runs in float32 (float64 accumulation rounded to float32), and the final
  Q is rounded to bfloat16 before Y = Q X0, whose result is rounded to
  bfloat16.  Reason: R <- P R P squares the singular values, so a bfloat16
  R cannot resolve singular values below about 2^-4 of the largest and the
  recurrence amplifies its rounding by up to a^2 ~ 12 per step; the pages
  give gram no precision, and FP32 for the small m x m recurrence is the
  reading that keeps gram as accurate as the standard method.
"""
import numpy as np

from .bf16 import round_bf16

A_COEF, B_COEF, C_COEF = 3.4445, -4.7750, 2.0315
DEFAULT_STEPS = 5
NORM_EPS = 1e-7

# Number of Newton-Schulz invocations since the last reset.  The pages count
# NS calls per optimizer step ("Run Muon once per optimizer step under
# ZeRO-3, not once per micro-batch", "The problem" table and "Testing").
NS_CALLS = [0]


def quintic(x):
    """f(x) = a x + b x^3 + c x^5, the scalar map NS applies to each
    singular value of the normalised input."""
    return A_COEF * x + B_COEF * x ** 3 + C_COEF * x ** 5


# ---------------------------------------------------------------- helpers

def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _gemm_bf16(lhs, rhs, alpha, E=None, beta=0.0, gamma=0.0):
    """bf16(alpha*(lhs @ rhs) + beta*E + gamma*I): product accumulated in
    float64, rounded to float32, epilogue in float32, result in bfloat16."""
    acc = _f32(np.asarray(lhs, np.float64) @ np.asarray(rhs, np.float64))
    out = np.float32(alpha) * acc
    if E is not None:
        out = out + np.float32(beta) * _f32(E)
    if gamma != 0.0:
        d = np.arange(min(out.shape))
        out[d, d] = out[d, d] + np.float32(gamma)
    return round_bf16(_f32(out))


def normalise(G, mode, eps=NORM_EPS):
    """X0 = G / (||G||_F + eps).

    exact: float64 throughout.  bf16 / fp32 storage: the sum of squares is
    taken in float64, the divisor d = sqrt(sum) + eps is rounded to float32,
    and X0 = G / d is a float32 division (then rounded to bfloat16 in bf16
    mode)."""
    if mode == "exact":
        G = np.asarray(G, np.float64)
        return G / (np.sqrt(np.sum(G * G)) + eps)
    G32 = _f32(G)
    s = np.sum(G32.astype(np.float64) ** 2)
    d = np.float32(np.sqrt(s) + eps)
    X0 = G32 / d
    return round_bf16(X0) if mode == "bf16" else X0


def _standard(X, steps, mode):
    a, b, c = A_COEF, B_COEF, C_COEF
    for _ in range(steps):
        if mode == "exact":
            A = X @ X.T
            B = b * A + c * (A @ A)
            X = a * X + B @ X
        else:
            A = _gemm_bf16(X, X.T, 1.0)
            B = _gemm_bf16(A, A, c, A, b)
            X = _gemm_bf16(B, X, 1.0, X, a)
    return X


def _gemm_f32(lhs, rhs, alpha, E=None, beta=0.0, gamma=0.0):
    """float32(alpha*(lhs @ rhs) + beta*E + gamma*I): product accumulated in
    float64, rounded to float32, epilogue in float32, result kept float32."""
    acc = _f32(np.asarray(lhs, np.float64) @ np.asarray(rhs, np.float64))
    out = np.float32(alpha) * acc
    if E is not None:
        out = out + np.float32(beta) * _f32(E)
    if gamma != 0.0:
        d = np.arange(min(out.shape))
        out[d, d] = out[d, d] + np.float32(gamma)
    return _f32(out)


def _gram(X0, steps, mode):
    a, b, c = A_COEF, B_COEF, C_COEF
    m = X0.shape[0]
    if mode == "exact":
        R = X0 @ X0.T
        Q = np.eye(m)
        for k in range(steps):
            P = a * np.eye(m) + b * R + c * (R @ R)
            Q = P @ Q
            if k < steps - 1:
                R = (P @ R) @ P
        return Q @ X0
    R = _gemm_f32(X0, X0.T, 1.0)
    Q = None
    for k in range(steps):
        P = _gemm_f32(R, R, c, R, b, gamma=a)
        Q = P if k == 0 else _gemm_f32(P, Q, 1.0)   # Q0 = I, so Q1 = P
        if k < steps - 1:
            T = _gemm_f32(P, R, 1.0)
            R = _gemm_f32(T, P, 1.0)
    return _gemm_bf16(round_bf16(Q), X0, 1.0)


def iterate(X0, method="standard", steps=DEFAULT_STEPS, mode="exact"):
    """Run the NS iteration on an already normalised X0 (any orientation);
    returns the result in X0's orientation."""
    if method not in ("standard", "gram"):
        raise ValueError(f"unknown ns method {method!r}")
    if steps < 1:
        raise ValueError("ns steps must be >= 1")
    X0 = np.asarray(X0, np.float64 if mode == "exact" else np.float32)
    transposed = X0.shape[0] > X0.shape[1]
    X = X0.T.copy() if transposed else X0
    Y = _standard(X, steps, mode) if method == "standard" else _gram(X, steps, mode)
    return Y.T.copy() if transposed else Y


def newton_schulz(G, method="standard", steps=DEFAULT_STEPS, mode="exact"):
    """Orthogonalise one matrix: normalise, orient so rows <= cols, iterate,
    transpose back.  Counts one NS call."""
    NS_CALLS[0] += 1
    return iterate(normalise(G, mode), method, steps, mode)
