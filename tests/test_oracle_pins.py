"""Pins for the CPU oracle: each test checks the oracle against something
that does not come from the oracle itself -- an SVD closed form, calculus
facts about the quintic, torch's bfloat16 conversion, numbers the pages
print (tests/golden/), brute force on tiny inputs, or an invariant the pages
state.  A few tests plant a mistake in the oracle (on the CPU) and check
that a pin catches it."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import bf16 as obf
from oracle import muon as om
from oracle import newton_schulz as ons
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# The quintic's coefficients are an assumption (the standard Muon values);
# the tests write the scalar map out on their own, in Horner form.
def f_scalar(x):
    x2 = x * x
    return x * (3.4445 + x2 * (-4.7750 + x2 * 2.0315))


def svd_closed_form(G, steps=5, eps=1e-7):
    """NS(G) = U f^steps(S / (||G||_F + eps)) V^T from a brute-force SVD."""
    G = np.asarray(G, np.float64)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    s = S / (np.linalg.norm(G) + eps)
    for _ in range(steps):
        s = f_scalar(s)
    return (U * s) @ Vt


def relf(a, b):
    return np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-300)


SHAPES = [(1, 7), (5, 1), (3, 3), (13, 17), (17, 13), (9, 17), (40, 24), (64, 96)]


# ------------------------------------------------------------ bfloat16

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(20000).astype(np.float32) * 1e3,
            rng.standard_normal(2000).astype(np.float32) * 1e-39,   # subnormals
            np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                      1.0, 1.00390625, 1.01171875], np.float32)]
    # exact ties: low 16 bits 0x8000 with even and odd kept bit
    ties = (np.arange(1, 4000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate(vals + [ties, -ties])
    mine = obf.round_bf16(x).view(np.uint32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().view(np.uint32)
    assert np.array_equal(mine, ref)
    assert np.all(mine & 0xFFFF == 0)


def test_bf16_rejects_wider_input():
    with pytest.raises(TypeError):
        obf.round_bf16(np.ones(3))


# ------------------------------------------------------------ the quintic

def test_quintic_critical_points_and_band():
    # f'(x) = a + 3b x^2 + 5c x^4 = 0 solved as a quadratic in x^2
    a, b, c = 3.4445, -4.7750, 2.0315
    disc = (3 * b) ** 2 - 4 * (5 * c) * a
    r = sorted([(-3 * b - np.sqrt(disc)) / (10 * c), (-3 * b + np.sqrt(disc)) / (10 * c)])
    xmax, xmin = np.sqrt(r[0]), np.sqrt(r[1])
    assert abs(xmax - 0.5545) < 1e-3 and abs(xmin - 1.0502) < 1e-3
    assert abs(ons.quintic(xmax) - 1.2024) < 1e-3
    assert abs(ons.quintic(xmin) - 0.6818) < 1e-3
    # f maps the band [0.6818, 1.2024] into itself
    xs = np.linspace(0.6818, 1.2024, 10001)
    ys = ons.quintic(xs)
    assert ys.min() >= 0.6818 - 1e-4 and ys.max() <= 1.2024 + 1e-4
    # slope at zero a: the pages' 'fifth power of its slope at zero'
    # ("Fix Muon optimizer under ZeRO CPU offload ...", fp16-noise commit)
    assert abs(a ** 5 - 485.0) < 1.0


# ------------------------------------------------------------ NS, exact

@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("shape", SHAPES)
def test_ns_exact_matches_svd_closed_form(method, shape):
    G = wl.rng_for(11, *shape).standard_normal(shape)
    Y = ons.newton_schulz(G, method, 5, "exact")
    assert Y.shape == G.shape
    assert relf(Y, svd_closed_form(G)) < 1e-10


@pytest.mark.parametrize("steps", [1, 2, 3, 7])
def test_ns_exact_step_count(steps):
    G = wl.rng_for(12).standard_normal((11, 19))
    for method in ("standard", "gram"):
        assert relf(ons.newton_schulz(G, method, steps, "exact"),
                    svd_closed_form(G, steps)) < 1e-10


def test_ns_zero_matrix_gives_zero():
    for method in ("standard", "gram"):
        for mode in ("exact", "bf16"):
            Y = ons.newton_schulz(np.zeros((4, 6), np.float32), method, 5, mode)
            assert np.all(Y == 0)


def test_ns_singular_values_in_band():
    # normalised Gaussian 17x13 and 9x17 (the tiny case's shapes): all
    # singular values land in the quintic's invariant band after 5 steps
    for shape in [(17, 13), (9, 17)]:
        G = wl.rng_for(13, *shape).standard_normal(shape)
        s = np.linalg.svd(ons.newton_schulz(G, "standard"), compute_uv=False)
        assert s.min() >= 0.6818 - 1e-6 and s.max() <= 1.2024 + 1e-6
        # singular vectors: Y and U V^T share their polar factor
        U, _, Vt = np.linalg.svd(G, full_matrices=False)
        Uy, _, Vty = np.linalg.svd(ons.newton_schulz(G, "standard"), full_matrices=False)
        assert relf(Uy @ Vty, U @ Vt) < 1e-8


def test_transpose_equivariance_exact_bits():
    for shape in [(13, 17), (9, 17), (40, 24)]:
        G = wl.rng_for(14, *shape).standard_normal(shape).astype(np.float32)
        for method in ("standard", "gram"):
            for mode in ("exact", "bf16"):
                a = ons.newton_schulz(G, method, 5, mode)
                b = ons.newton_schulz(G.T.copy(), method, 5, mode)
                assert np.array_equal(a, b.T)


def test_gram_equals_standard_exact():
    G = wl.rng_for(15).standard_normal((24, 70))
    assert relf(ons.newton_schulz(G, "gram"), ons.newton_schulz(G, "standard")) < 1e-12


# ------------------------------------------------------------ NS, bf16 mode

@pytest.mark.parametrize("method", ["standard", "gram"])
def test_bf16_mode_within_bf16_noise_of_closed_form(method):
    for shape in [(17, 13), (9, 17), (64, 96), (32, 128)]:
        G = wl.rng_for(16, *shape).standard_normal(shape).astype(np.float32)
        Y = ons.newton_schulz(G, method, 5, "bf16")
        assert Y.dtype == np.float32
        assert np.all(Y.view(np.uint32) & 0xFFFF == 0), "outputs must be bf16 values"
        err = relf(Y, svd_closed_form(G))
        assert 1e-4 < err < 4e-2, err     # bf16 noise: present, but small


def _rne_bf16_scalar(v):
    """Round one float32 to bfloat16 by hand: bits via tobytes."""
    u = int(np.float32(v).view(np.uint32))
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return float(np.uint32(u).view(np.float32))


def test_bf16_mode_one_step_brute_force():
    """One standard step on a 2x3 matrix, written as scalar loops with the
    rounding points (X0, A, B, X) and the float32 epilogue order."""
    G = np.array([[0.3, -1.2, 0.7], [2.0, 0.1, -0.4]], np.float32)
    a, b, c = 3.4445, -4.7750, 2.0315
    f32 = np.float32
    d = f32(np.sqrt(float(np.sum(G.astype(np.float64) ** 2))) + 1e-7)
    X = [[_rne_bf16_scalar(f32(G[i, j]) / d) for j in range(3)] for i in range(2)]
    A = [[_rne_bf16_scalar(f32(sum(X[i][k] * X[j][k] for k in range(3)))) for j in range(2)]
         for i in range(2)]
    B = [[_rne_bf16_scalar(f32(f32(c) * f32(sum(A[i][k] * A[k][j] for k in range(2))))
                           + f32(f32(b) * f32(A[i][j]))) for j in range(2)] for i in range(2)]
    X1 = [[_rne_bf16_scalar(f32(f32(sum(B[i][k] * X[k][j] for k in range(2))))
                            + f32(f32(a) * f32(X[i][j]))) for j in range(3)] for i in range(2)]
    Y = ons.newton_schulz(G, "standard", 1, "bf16")
    assert np.array_equal(Y, np.array(X1, np.float32))


def _gram_bf16_brute(G, steps, r_in_bf16=False, q_to_bf16=True):
    """The gram method in BF16-operand mode written as scalar loops, with
    the rounding points of the reading: X0 = bf16(G / d); R0 = fl32(sum of
    bf16 products); per step P = fl32(fl32(c * RR) + fl32(b * R)) (+ a on
    the diagonal, one more float32 addition), Q <- fl32(P Q) (Q1 = P),
    T = fl32(P R) and R = fl32(T P) except after the last step; finally
    Y = bf16(fl32(bf16(Q) X0)).  r_in_bf16 / q_to_bf16 switch the two
    rounding points a plausible mistake would move."""
    f32 = np.float32
    a, b, c = 3.4445, -4.7750, 2.0315
    m, n = G.shape
    assert m <= n
    d = f32(np.sqrt(float(np.sum(G.astype(np.float64) ** 2))) + 1e-7)
    X = [[_rne_bf16_scalar(f32(G[i, j]) / d) for j in range(n)] for i in range(m)]

    def rr(v):
        return _rne_bf16_scalar(v) if r_in_bf16 else v

    def prod(L, Rt, i, j, K):
        return f32(sum(float(L[i][k]) * float(Rt[k][j]) for k in range(K)))

    Xt = [[X[j][i] for j in range(m)] for i in range(n)]
    R = [[rr(prod(X, Xt, i, j, n)) for j in range(m)] for i in range(m)]
    Q = None
    for k in range(steps):
        P = []
        for i in range(m):
            row = []
            for j in range(m):
                v = f32(f32(f32(c) * prod(R, R, i, j, m)) + f32(f32(b) * f32(R[i][j])))
                if i == j:
                    v = f32(v + f32(a))
                row.append(v)
            P.append(row)
        Q = P if k == 0 else [[prod(P, Q, i, j, m) for j in range(m)] for i in range(m)]
        if k < steps - 1:
            T = [[prod(P, R, i, j, m) for j in range(m)] for i in range(m)]
            R = [[rr(prod(T, P, i, j, m)) for j in range(m)] for i in range(m)]
    Qy = [[_rne_bf16_scalar(q) if q_to_bf16 else q for q in row] for row in Q]
    return np.array([[_rne_bf16_scalar(prod(Qy, X, i, j, m)) for j in range(n)]
                     for i in range(m)], np.float32)


GRAM_BRUTE_CASES = [(np.array([[0.3, -1.2, 0.7], [2.0, 0.1, -0.4]], np.float32), 1),
                    (np.array([[0.3, -1.2, 0.7], [2.0, 0.1, -0.4]], np.float32), 2),
                    (wl.rng_for(31).standard_normal((3, 5)).astype(np.float32), 1),
                    (wl.rng_for(31).standard_normal((3, 5)).astype(np.float32), 2),
                    (wl.rng_for(32).standard_normal((3, 5)).astype(np.float32), 3)]


@pytest.mark.parametrize("case", range(len(GRAM_BRUTE_CASES)))
def test_gram_bf16_mode_brute_force(case):
    """One, two and three gram steps on 2x3 and 3x5 matrices, scalar loops
    against the oracle, bit for bit (the BF16-mode gram reading: FP32
    recurrence, Q rounded to bf16 before Y)."""
    G, steps = GRAM_BRUTE_CASES[case]
    want = _gram_bf16_brute(G, steps)
    assert np.array_equal(ons.newton_schulz(G, "gram", steps, "bf16"), want)
    # the transposed input takes the same path (rows > cols is transposed)
    assert np.array_equal(ons.newton_schulz(G.T.copy(), "gram", steps, "bf16"), want.T)


def _planted_gram(r_in_bf16, q_to_bf16):
    """The oracle's BF16-mode gram with one rounding point moved."""
    def bad(X0, steps, mode):
        a, b, c = ons.A_COEF, ons.B_COEF, ons.C_COEF
        rr = (lambda M: obf.round_bf16(M)) if r_in_bf16 else (lambda M: M)
        R = rr(ons._gemm_f32(X0, X0.T, 1.0))
        Q = None
        for k in range(steps):
            P = ons._gemm_f32(R, R, c, R, b, gamma=a)
            Q = P if k == 0 else ons._gemm_f32(P, Q, 1.0)
            if k < steps - 1:
                R = rr(ons._gemm_f32(ons._gemm_f32(P, R, 1.0), P, 1.0))
        return ons._gemm_bf16(obf.round_bf16(Q) if q_to_bf16 else Q, X0, 1.0)
    return bad


@pytest.mark.parametrize("plant", [(True, True), (False, False)],
                         ids=["R kept in bf16", "Q not rounded before Y"])
def test_planted_gram_bf16_rounding_points_are_caught(monkeypatch, plant):
    monkeypatch.setattr(ons, "_gram", _planted_gram(*plant))
    caught = 0
    for G, steps in GRAM_BRUTE_CASES:
        caught += not np.array_equal(ons.newton_schulz(G, "gram", steps, "bf16"),
                                     _gram_bf16_brute(G, steps))
    assert caught >= 3


# ------------------------------------------------------------ planted mistakes

def test_planted_wrong_coefficient_sign_is_caught(monkeypatch):
    monkeypatch.setattr(ons, "B_COEF", +4.7750)
    G = wl.rng_for(17).standard_normal((9, 17))
    assert relf(ons.newton_schulz(G, "standard"), svd_closed_form(G)) > 1e-3


def test_planted_gram_missing_factor_is_caught(monkeypatch):
    def bad_gram(X0, steps, mode):
        a, b, c = ons.A_COEF, ons.B_COEF, ons.C_COEF
        R = X0 @ X0.T
        Q = np.eye(X0.shape[0])
        for k in range(steps):
            P = a * np.eye(len(R)) + b * R + c * R @ R
            Q = P @ Q
            R = P @ R          # planted: one factor of P dropped
        return Q @ X0
    monkeypatch.setattr(ons, "_gram", bad_gram)
    G = wl.rng_for(18).standard_normal((9, 17))
    assert relf(ons.newton_schulz(G, "gram"), svd_closed_form(G)) > 1e-3


def test_planted_missing_transpose_is_caught(monkeypatch):
    """Iterating a tall matrix without transposing it still approximates the
    polar factor in exact arithmetic, so the SVD pin cannot see it; the
    bit-exact transpose-equivariance pin does."""
    G = wl.rng_for(19).standard_normal((17, 13)).astype(np.float32)
    assert np.array_equal(ons.newton_schulz(G, "standard", 5, "bf16"),
                          ons.newton_schulz(G.T.copy(), "standard", 5, "bf16").T)

    def no_orient(X0, method="standard", steps=5, mode="exact"):
        return ons._standard(np.asarray(X0, np.float32), steps, mode)   # planted
    monkeypatch.setattr(ons, "iterate", no_orient)
    assert not np.array_equal(ons.newton_schulz(G, "standard", 5, "bf16"),
                              ons.newton_schulz(G.T.copy(), "standard", 5, "bf16").T)


def test_momentum_closed_form_and_planted_mistake(monkeypatch):
    g = np.full((3, 4), 0.5, np.float32)
    beta = 0.95

    def three_steps():
        m = np.zeros((3, 4), np.float32)
        for _ in range(3):
            m, _ = om.muon_update(g, m, beta, "standard")
        return m
    # three steps of m <- beta m + g from zero: g (1 + beta + beta^2)
    assert np.allclose(three_steps(), 0.5 * (1 + beta + beta ** 2), rtol=1e-6)
    monkeypatch.setattr(om, "momentum_update",
                        lambda m, g, b: np.float32(b) * m + np.float32(1 - b) * g)  # planted EMA
    assert not np.allclose(three_steps(), 0.5 * (1 + beta + beta ** 2), rtol=1e-3)


# ------------------------------------------------------------ Muon step

def _tiny_mats(layout, seed=1000, mode_bf16=True):
    mats = []
    for i, s in enumerate(layout.specs):
        rng = wl.rng_for(seed, i, 99)
        mats.append({"g": wl.to_bf16_values(rng.standard_normal((s.rows, s.cols)).astype(np.float32)),
                     "m": np.zeros((s.rows, s.cols), np.float32),
                     "w": (0.02 * rng.standard_normal((s.rows, s.cols))).astype(np.float32),
                     "use_muon": s.use_muon, "num_heads": s.num_heads})
    return mats


def test_tiny_layout_matches_hand_worked_golden():
    gold = golden("tiny_layout.json")
    lay = wl.tiny_layout()
    assert list(lay.params["offset"]) == gold["param_offsets"]
    assert [[int(q["flat_begin"]), int(q["flat_end"])] for q in lay.parts] == gold["partitions"]
    assert lay.flat_size == gold["flat_size"]
    # both Muon matrices are cut by a partition boundary
    for k in range(2):
        off = int(lay.params["offset"][k]); n = lay.specs[k].numel
        cuts = [int(q["flat_begin"]) for q in lay.parts if off < int(q["flat_begin"]) < off + n]
        assert cuts, f"matrix {k} not cut"


def test_page_fixed_ns_call_count():
    """2 matrices, 2 steps, gas=4: NS runs once per matrix per step."""
    gold = golden("page_facts.json")["ns_calls_two_matrices_two_steps_gas4"]
    specs = [wl.ParamSpec("a", 6, 10), wl.ParamSpec("b", 10, 6)]
    lay = wl.build_layout([specs], 16, 2)
    acc = np.zeros(lay.storage_size, np.float32)
    mom = np.zeros_like(acc)
    mst = np.zeros_like(acc)
    ons.NS_CALLS[0] = 0
    for step in range(2):
        for mb in range(4):
            g = wl.pack(lay, wl.gaussian_grads(lay, 5, step * 4 + mb))
            acc = om.accumulate(acc, g, 0.25, overwrite=(mb == 0))
        acc, mom, mst, res = om.muon_step_flat(acc, mom, mst, lay.params, lay.parts,
                                               0.95, 0.02, "gram", 5, 0.0, "exact")
    assert ons.NS_CALLS[0] == gold["value"]


def test_gas_equivalence_exact_sums():
    """gas=1 with the mean gradient and gas=4 with the four micro-batch
    gradients give bit-identical steps when the sums are exact ('Run Muon
    once per optimizer step ...', 'The problem': same samples either way)."""
    lay = wl.tiny_layout()
    rng = wl.rng_for(21)
    parts4 = [wl.pack(lay, [rng.integers(-64, 65, (s.rows, s.cols)) / 64.0 for s in lay.specs])
              for _ in range(4)]
    mean = wl.pack(lay, [np.zeros((s.rows, s.cols)) for s in lay.specs])
    for p in parts4:
        mean = mean + p
    mean = (mean / 4).astype(np.float32)
    acc1 = om.accumulate(None, mean, 1.0, overwrite=True)
    acc4 = None
    for i, p in enumerate(parts4):
        acc4 = om.accumulate(acc4, p, 0.25, overwrite=(i == 0))
    assert np.array_equal(acc1.view(np.uint32), acc4.view(np.uint32))
    z = np.zeros(lay.storage_size, np.float32)
    r1 = om.muon_step_flat(acc1, z, z, lay.params, lay.parts, 0.95, 0.02, "gram", 5, 0.05, "bf16")
    r4 = om.muon_step_flat(acc4, z, z, lay.params, lay.parts, 0.95, 0.02, "gram", 5, 0.05, "bf16")
    for a, b in zip(r1[:3], r4[:3]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("mode", ["exact", "bf16"])
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_partition_independence_and_padding(mode, method):
    """Flat path with P=1, 2, 8, rank-major and shuffled storage equals the
    full-matrix reference with no tables at all, bit for bit; padding and
    gaps keep their sentinel bits ('Support Muon in BF16_Optimizer ...',
    validation table: 17x13 / 9x17 crossing partitions match an
    independent full-matrix reference exactly)."""
    base = wl.tiny_layout()
    mats = _tiny_mats(base)
    ref = om.muon_step_full(mats, 0.95, 0.02, method, 5, 0.05, mode)
    for nparts, storage in [(1, "identity"), (2, "identity"), (8, "identity"),
                            (2, "rank_major"), (8, "shuffled")]:
        lay = wl.tiny_layout(nparts, storage, seed=nparts)
        acc = wl.storage_with_sentinels(lay, [d["g"] for d in mats])
        mom = wl.storage_with_sentinels(lay, [d["m"] for d in mats])
        mst = wl.storage_with_sentinels(lay, [d["w"] for d in mats])
        a2, m2, w2, res = om.muon_step_flat(acc, mom, mst, lay.params, lay.parts,
                                            0.95, 0.02, method, 5, 0.05, mode)
        pad = wl.padding_mask(lay)
        for before, after, key in [(acc, a2, "update"), (mom, m2, "momentum"), (mst, w2, "master")]:
            assert np.array_equal(before.view(np.uint32)[pad], after.view(np.uint32)[pad])
            got = wl.unpack(lay, after)
            for k, spec in enumerate(lay.specs):
                want = ref[key][k]
                assert np.array_equal(got[k].view(np.uint32), np.asarray(want, np.float32).view(np.uint32)), (nparts, storage, key, k)
        assert res["norm"] == ref["norm"] and res["coef"] == ref["coef"]


def test_global_norm_and_clip_against_svd():
    lay = wl.tiny_layout()
    mats = _tiny_mats(lay)
    res = om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 0.05, "exact")
    sq = 0.0
    for d in mats:
        if d["use_muon"]:
            sq += np.sum(svd_closed_form(0.95 * d["m"] + d["g"]) ** 2)   # m0 = 0
        else:
            sq += np.sum(np.asarray(d["g"], np.float64) ** 2)
    assert abs(res["norm"] - np.sqrt(sq)) < 1e-9 * np.sqrt(sq)
    assert abs(res["coef"] - 0.05 / (np.sqrt(sq) + 1e-6)) < 1e-12
    # clip larger than the norm: no scaling; clip <= 0: disabled
    assert om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 1e6, "exact")["coef"] == 1.0
    assert om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 0.0, "exact")["coef"] == 1.0
    # the aux update is the clipped gradient; its master is untouched
    assert np.allclose(res["update"][2], res["coef"] * mats[2]["g"], rtol=1e-6)
    assert np.array_equal(res["master"][2], mats[2]["w"])
    # Muon master moves by -lr * update
    assert np.allclose(res["master"][0], mats[0]["w"] - 0.02 * res["update"][0], atol=1e-8)


def test_overflow_skips_step_and_keeps_momentum():
    lay = wl.tiny_layout()
    mats = _tiny_mats(lay)
    mats[1]["g"] = mats[1]["g"].copy()
    mats[1]["g"][3, 4] = np.inf
    acc = wl.storage_with_sentinels(lay, [d["g"] for d in mats])
    mom = wl.storage_with_sentinels(lay, [np.full_like(d["g"], 0.25) for d in mats])
    mst = wl.storage_with_sentinels(lay, [d["w"] for d in mats])
    a2, m2, w2, res = om.muon_step_flat(acc, mom, mst, lay.params, lay.parts, 0.95, 0.02)
    assert res["applied"] == 0 and res["ns_calls"] == 0
    for x, y in [(acc, a2), (mom, m2), (mst, w2)]:
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    # a NaN in padding is not an overflow
    acc_ok = wl.storage_with_sentinels(lay, [d["g"] if k != 1 else np.zeros_like(d["g"])
                                             for k, d in enumerate(mats)])
    assert om.muon_step_flat(acc_ok, mom, mst, lay.params, lay.parts, 0.95, 0.02)[3]["applied"] == 1


def test_per_head_blocks_match_svd_and_leave_untagged_alone():
    gold = golden("page_facts.json")["per_head"]
    rng = wl.rng_for(22)
    q = rng.standard_normal((12, 8)).astype(np.float32)
    mlp = rng.standard_normal((8, 12)).astype(np.float32)
    z = lambda x: np.zeros_like(x)
    mk = lambda heads: [{"g": q, "m": z(q), "w": z(q), "use_muon": True, "num_heads": heads},
                        {"g": mlp, "m": z(mlp), "w": z(mlp), "use_muon": True, "num_heads": 0}]
    whole = om.muon_step_full(mk(0), 0.9, 0.1, "standard", 5, 0.0, "exact")
    heads = om.muon_step_full(mk(3), 0.9, 0.1, "standard", 5, 0.0, "exact")
    assert "q" in gold["changes"] and "mlp" in gold["unchanged"]
    assert relf(heads["update"][0], whole["update"][0]) > 1e-2          # q moves
    assert np.array_equal(heads["update"][1], whole["update"][1])       # mlp does not
    for h in range(3):   # each 4x8 head block is its own NS problem
        blk = heads["update"][0][4 * h:4 * (h + 1)].astype(np.float64)
        assert relf(blk, svd_closed_form(q[4 * h:4 * (h + 1)])) < 1e-6
    assert heads["ns_calls"] == 4 and whole["ns_calls"] == 2


def test_bad_tables_raise():
    lay = wl.tiny_layout()
    acc = np.zeros(lay.storage_size, np.float32)
    bad = lay.params.copy()
    bad["offset"][0] = lay.flat_size - 10        # runs past the partitions
    with pytest.raises(ValueError):
        om.muon_step_flat(acc, acc, acc, bad, lay.parts, 0.95, 0.02)


def _f32_round(x):
    """Nearest float32 of a Python float (IEEE round to nearest even), by
    the C library's double -> float conversion inside struct."""
    import struct
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_accumulate_rounding_sequence():
    """Each micro-batch adds fl32(fl32(scale) * g) to the FP32 accumulator
    with one FP32 rounding per operation.  The expected values come from
    Python floats (exact here: products of two float32 values and sums of
    two close float32 values fit a double) rounded to float32 by struct,
    not from numpy."""
    g1 = wl.to_bf16_values(wl.rng_for(33).standard_normal(64).astype(np.float32))
    g2 = wl.to_bf16_values(wl.rng_for(34).standard_normal(64).astype(np.float32))
    s32 = _f32_round(1.0 / 3.0)
    want_a = [_f32_round(s32 * float(x)) for x in g1]
    a = om.accumulate(None, g1, 1.0 / 3.0, overwrite=True)
    assert a.tolist() == want_a
    want_b = [_f32_round(x + _f32_round(s32 * float(y))) for x, y in zip(want_a, g2)]
    b = om.accumulate(a, g2, 1.0 / 3.0)
    assert b.tolist() == want_b
    # the inputs tell the two roundings apart: a fused multiply-add (the
    # product left unrounded) gives other values on some elements
    fused = [_f32_round(x + s32 * float(y)) for x, y in zip(want_a, g2)]
    assert sum(u != v for u, v in zip(want_b, fused)) >= 5
