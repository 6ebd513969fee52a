"""The Newton-Schulz sweep at its full sizes (8192^2, 16384^2, 4096x16384,
16384x4096; X ~ N(0,1), bf16 for BF16 operands), through the same entry
point and launch configuration the sweep bench times.  The oracle cannot
run these sizes on the host, so they are checked through properties that
hold at any size:

* the step map, by Freivalds' probe: for a random vector v,
  X_{k+1} v = a X_k v + b A X_k v + c A^2 X_k v with A = X_k X_k^T
  (canonical orientation, rows <= cols), evaluated with fp64
  matrix-vector products.  X_k is the k-step output of the entry: the entry
  is deterministic, so the k- and (k+1)-step runs share their first k
  steps, and the standard form keeps every iterate in the output format
  (bf16 in BF16 mode, exact split-3 in FP32 mode), so the k-step output is
  the iterate itself.  The gram form equals the standard one in exact
  arithmetic, so its k-step outputs obey the same map within rounding.
  Step 0 -> 1 starts from X_0 = G / (||G||_F + 1e-7) formed here in fp64
  (rounded to bf16 in BF16 mode, as the entry does).
* the band: every singular value of the result stays below the quintic's
  local maximum f(0.5545) = 1.2024 (power iteration on Y^T Y in fp64); for
  the wide 4096 x 16384 Gaussian, whose normalised singular values lie
  near [0.5, 1.5] / 64, well above 2.69e-3, all of them end inside
  [0.6818, 1.2024] (eigenvalues of Y Y^T).

Tolerances: the probe compares a result rounded at every product (BF16:
A, B and X rounded to bf16, relative 2^-9 each, over terms of size up to
|b|, |c| ~ 5 that cancel to ~1) with exact arithmetic on the same X_k;
3e-2 relative in BF16 mode, 1e-4 in FP32 mode for the standard form
(split-3 products carry ~1e-6, and X_k is the very iterate X_{k+1} was made
from).  The gram form's k- and (k+1)-step outputs come from separate runs
of the recurrence (Q_k X0 is formed anew each run), so the probe sees both
runs' rounding, amplified by up to a = 3.4 through the step map; its FP32
bound is the FP32 parity rule's rtol, 1e-3 (the compiled-NS check of
"Support Muon in BF16_Optimizer with FP32 gradient accumulation",
validation table).  A wrong coefficient, a dropped term or a transposed
operand moves the probe by O(1).  Band edges get 2% (BF16) / 1e-4 (FP32)."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import oracle.newton_schulz as ons
import workloads as wl

pytestmark = pytest.mark.gpu

A, B, C = ons.A_COEF, ons.B_COEF, ons.C_COEF
F_MAX, F_MIN = 1.2024, 0.6818       # quintic's local max f(0.5545), local min f(1.0501)
PROBE_TOL = {("bf16", "standard"): 3e-2, ("bf16", "gram"): 3e-2,
             ("fp32", "standard"): 1e-4, ("fp32", "gram"): 1e-3}
BAND_TOL = {"bf16": 2e-2, "fp32": 1e-4}


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def sweep_input(torch, r, c, mode, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    X = torch.randn((r, c), generator=gen, device="cuda", dtype=torch.float32)
    return X.to(torch.bfloat16) if mode == "bf16" else X


def canon64(torch, Y):
    """fp64 copy in canonical orientation (rows <= cols)."""
    Y = Y.to(torch.float64)
    return Y.t().contiguous() if Y.shape[0] > Y.shape[1] else Y


def step_probe(X, v):
    """a X v + b A X v + c A^2 X v, A = X X^T, by matrix-vector products."""
    u0 = X @ v
    u1 = X @ (X.t() @ u0)
    u2 = X @ (X.t() @ u1)
    return A * u0 + B * u1 + C * u2


def probe_error(torch, X_k, X_next, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    worst = 0.0
    for _ in range(2):
        v = torch.randn(X_k.shape[1], generator=gen, device="cuda", dtype=torch.float64)
        ref = step_probe(X_k, v)
        got = X_next @ v
        worst = max(worst, float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref)))
    return worst


def sigma_max(torch, Y, iters=60):
    gen = torch.Generator(device="cuda").manual_seed(5)
    w = torch.randn(Y.shape[1], generator=gen, device="cuda", dtype=torch.float64)
    for _ in range(iters):
        w = Y.t() @ (Y @ w)
        w = w / torch.linalg.norm(w)
    return float(torch.linalg.norm(Y @ w))


CASES = [
    # rows, cols, method, mode
    (8192, 8192, "standard", "bf16"),
    (8192, 8192, "gram", "bf16"),
    (8192, 8192, "standard", "fp32"),
    (8192, 8192, "gram", "fp32"),
    (16384, 16384, "standard", "bf16"),
    (16384, 16384, "gram", "bf16"),
    (16384, 16384, "standard", "fp32"),
    (16384, 16384, "gram", "fp32"),
    (4096, 16384, "standard", "bf16"),
    (4096, 16384, "gram", "bf16"),
    (4096, 16384, "gram", "fp32"),
    (4096, 16384, "standard", "fp32"),
    (16384, 4096, "standard", "bf16"),
    (16384, 4096, "standard", "fp32"),
    (16384, 4096, "gram", "bf16"),
    (16384, 4096, "gram", "fp32"),
]


@pytest.mark.parametrize("rows,cols,method,mode", CASES)
def test_full_size_step_map_and_band(torch, rows, cols, method, mode):
    X = sweep_input(torch, rows, cols, mode, wl.CONFIG_SEED["sweep"] + rows + 3 * cols)
    outs = {}
    for k in (1, 4, 5):
        Y = torch.empty_like(X)
        nsg.newton_schulz(X, Y, method, k, mode)
        outs[k] = canon64(torch, Y)
    torch.cuda.synchronize()
    assert nsg.device_error() == 0
    tol = PROBE_TOL[(mode, method)]
    # step 0 -> 1 from X_0 formed here
    G = canon64(torch, X)
    X0 = G / (torch.linalg.norm(G) + 1e-7)
    if mode == "bf16":
        X0 = X0.to(torch.bfloat16).to(torch.float64)
    e01 = probe_error(torch, X0, outs[1], 11)
    e45 = probe_error(torch, outs[4], outs[5], 12)
    print(f"{rows}x{cols} {method} {mode}: probe 0->1 {e01:.2e}, 4->5 {e45:.2e}")
    assert e01 <= tol, (e01, tol)
    assert e45 <= tol, (e45, tol)
    # band: nothing above the quintic's local maximum
    smax = sigma_max(torch, outs[5])
    assert smax <= F_MAX * (1 + BAND_TOL[mode]), smax
    if (rows, cols) == (4096, 16384):
        s = torch.linalg.eigvalsh(outs[5] @ outs[5].t()).clamp_min(0).sqrt()
        lo, hi = float(s.min()), float(s.max())
        print(f"  singular values in [{lo:.4f}, {hi:.4f}]")
        assert lo >= F_MIN * (1 - BAND_TOL[mode]) and hi <= F_MAX * (1 + BAND_TOL[mode]), (lo, hi)
