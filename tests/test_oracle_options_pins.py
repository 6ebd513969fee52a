"""Pins for the oracle's step options: the gradient-clipping order, the
loss-scale undo and the fused auxiliary Adam update.  Each is checked
against something outside the oracle: torch.optim.Adam, exact power-of-two
scaling, an independent norm, the SVD closed form of NS."""
import numpy as np
import pytest

from oracle import muon as om
from oracle import newton_schulz as ons
import workloads as wl

from test_oracle_pins import svd_closed_form, relf


def _mats(seed=3):
    lay = wl.tiny_layout()
    out = []
    for i, s in enumerate(lay.specs):
        rng = wl.rng_for(seed, i)
        d = {"g": wl.to_bf16_values(rng.standard_normal((s.rows, s.cols)).astype(np.float32)),
             "m": np.zeros((s.rows, s.cols), np.float32),
             "w": (0.1 * rng.standard_normal((s.rows, s.cols))).astype(np.float32),
             "use_muon": s.use_muon, "num_heads": 0}
        if not s.use_muon:
            d["exp_avg"] = np.zeros((s.rows, s.cols), np.float32)
            d["exp_avg_sq"] = np.zeros((s.rows, s.cols), np.float32)
        out.append(d)
    return out


def test_adam_matches_torch_optim_adam():
    torch = pytest.importorskip("torch")
    rng = wl.rng_for(5)
    w0 = rng.standard_normal((8, 5)).astype(np.float32)
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([p], lr=1e-3, betas=(0.9, 0.999), eps=1e-8)
    m = np.zeros_like(w0)
    v = np.zeros_like(w0)
    w = w0.copy()
    for t in range(1, 6):
        g = rng.standard_normal((8, 5)).astype(np.float32)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        m, v, w = om.adam_update(g, m, v, w, 1e-3, 0.9, 0.999, 1e-8, t)
        st = opt.state[p]
        # torch forms the first moment as a lerp, m + (1 - b1)(g - m), which
        # rounds differently from b1 m + (1 - b1) g from step 2 on
        assert np.allclose(m, st["exp_avg"].numpy(), rtol=1e-5, atol=1e-8)
        assert np.allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-12)
        assert np.allclose(w, p.detach().numpy(), rtol=1e-6, atol=1e-8)


def test_planted_adam_without_bias_correction_is_caught():
    torch = pytest.importorskip("torch")
    w0 = np.ones((3, 3), np.float32)
    g = np.full((3, 3), 0.5, np.float32)
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([p], lr=1e-2)
    p.grad = torch.from_numpy(g.copy())
    opt.step()
    _, _, w_ok = om.adam_update(g, 0 * g, 0 * g, w0, 1e-2, 0.9, 0.999, 1e-8, 1)
    _, _, w_bad = om.adam_update(g, 0 * g, 0 * g, w0, 1e-2, 0.9, 0.999, 1e-8, 10 ** 9)  # planted
    assert np.allclose(w_ok, p.detach().numpy(), rtol=1e-6)
    assert not np.allclose(w_bad, p.detach().numpy(), rtol=1e-3)


@pytest.mark.parametrize("clip_mode", ["update", "grad"])
def test_loss_scale_undo_is_exact(clip_mode):
    """accum = 2^12 * g with grad_scale 2^-12 gives bit-identical results to
    accum = g: power-of-two scaling is exact, so the norm never sees the
    loss scale."""
    base = _mats()
    scaled = [dict(d, g=np.float32(4096.0) * d["g"]) for d in base]
    adam = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=1)
    a = om.muon_step_full(base, 0.95, 0.02, "gram", 5, 0.05, "bf16", clip_mode, 1.0, adam)
    b = om.muon_step_full(scaled, 0.95, 0.02, "gram", 5, 0.05, "bf16", clip_mode, 2.0 ** -12, adam)
    assert a["norm"] == b["norm"] and a["coef"] == b["coef"]
    for key in ("update", "momentum", "master", "exp_avg", "exp_avg_sq"):
        for x, y in zip(a[key], b[key]):
            if x is not None:
                assert np.array_equal(np.asarray(x).view(np.uint32), np.asarray(y).view(np.uint32))


def test_pre_clip_norm_and_scale_invariance():
    """clip_mode 'grad': the norm is over all gradients; Muon's update of the
    clipped gradient equals NS of the clipped gradient (closed form), and
    with zero momentum it hardly depends on the clip at all (NS normalises);
    auxiliary updates are the clipped gradient."""
    mats = _mats()
    res = om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 0.05, "exact", "grad")
    allg = np.concatenate([np.asarray(d["g"], np.float64).ravel() for d in mats])
    norm = np.linalg.norm(allg)
    assert abs(res["norm"] - norm) < 1e-12 * norm
    coef = 0.05 / (norm + 1e-6)
    assert abs(res["coef"] - coef) < 1e-15
    for d, u in zip(mats, res["update"]):
        if d["use_muon"]:
            g_c = np.float32(coef) * d["g"]
            assert relf(u, svd_closed_form(g_c)) < 1e-6
            assert relf(u, svd_closed_form(d["g"])) < 1e-5       # scale invariance
        else:
            assert np.array_equal(u, np.float32(coef) * d["g"])
    # the Muon master moves by -lr * u (no second scaling)
    assert np.allclose(res["master"][0], mats[0]["w"] - 0.02 * res["update"][0], atol=1e-8)
    # clip above the norm: the pre-clip step equals the post-clip step
    a = om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 1e9, "exact", "grad")
    b = om.muon_step_full(mats, 0.95, 0.02, "standard", 5, 1e9, "exact", "update")
    for x, y in zip(a["update"], b["update"]):
        assert np.array_equal(x, y)
