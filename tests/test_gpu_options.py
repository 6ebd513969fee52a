"""Parity of muon_step_ex's options with the oracle: clipping the gradients
before Muon, undoing a loss scale, and the fused Adam step of the auxiliary
parameters.

Tolerances, beyond the rules in ``harness``:
* the clip coefficient is a float formed from a sum of squares whose
  summation order differs between the two sides, so it may differ in its
  last bit; quantities scaled by it are compared at 1e-6 relative to the
  magnitude of their terms (the auxiliary write-back coef g; the momentum
  beta m + coef g, against |beta m| + |coef g|), and bit-exactly wherever
  the coefficient is exactly 1;
* Adam is elementwise FP32 arithmetic in the same operation order on both
  sides: bit-exact when its input gradient is (coefficient 1), else
  rtol 1e-5 (one coefficient ulp through the moment updates);
* a power-of-two grad_scale is exact, so a scaled gradient with the
  reciprocal grad_scale reproduces the unscaled step bit for bit."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import oracle.muon as om
import workloads as wl
from harness import ORACLE_MODE, GpuState, assert_close_update, bits, to_dev

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05
# FP32-exact hyperparameters, so the oracle (double Python floats) and the
# library (float arguments) see the same values
F = lambda x: float(np.float32(x))   # noqa: E731
ADAM = dict(lr=F(1e-3), beta1=F(0.9), beta2=F(0.999), eps=F(1e-8))


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def mixed_layout(nparts=3, storage="identity", seed=0):
    """Muon matrices in both orientations, one split into 4 heads, and
    auxiliary groups of aligned (LayerNorm-like rows, an embedding-like
    block) and ragged (7x5) sizes; 128-element alignment."""
    return wl.build_layout(
        [[wl.ParamSpec("wq", 128, 192, 4), wl.ParamSpec("wt", 192, 128)],
         [wl.ParamSpec("ln", 1, 768, use_muon=False), wl.ParamSpec("emb", 40, 768, use_muon=False)],
         [wl.ParamSpec("odd", 7, 5, use_muon=False), wl.ParamSpec("w17", 17, 13)]], 128, nparts,
        storage, seed)


def make_state(torch, lay, seed, scale=1.0, adam=False):
    g = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-3, 1e-1))
    g = [np.float32(scale) * x for x in g]
    m = [np.float32(0.01) * x for x in wl.gaussian_grads(lay, seed, 1, None, bf16=False)]
    w = wl.gaussian_grads(lay, seed, 2, None, bf16=False)
    st = GpuState(torch, wl.storage_with_sentinels(lay, g), wl.storage_with_sentinels(lay, m),
                  wl.storage_with_sentinels(lay, w))
    if adam:
        z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
        st.exp_avg = to_dev(wl.storage_with_sentinels(lay, z), torch)
        st.exp_avg_sq = to_dev(wl.storage_with_sentinels(lay, z), torch)
    return st


def adam_dict(st, step):
    return dict(ADAM, step=step, exp_avg=st.exp_avg, exp_avg_sq=st.exp_avg_sq)


def muon_mask(lay):
    return wl.pack(lay, [np.full((s.rows, s.cols), 1 if s.use_muon else 0, np.int8)
                         for s in lay.specs], np.int8, 0).astype(bool)


def aux_mask(lay):
    return wl.pack(lay, [np.full((s.rows, s.cols), 0 if s.use_muon else 1, np.int8)
                         for s in lay.specs], np.int8, 0).astype(bool)


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
@pytest.mark.parametrize("lay_name", ["tiny", "mixed"])
def test_gradient_clip_before_muon(torch, method, mode, lay_name):
    """clip_mode grad: the norm is the gradient norm, the momentum takes the
    clipped gradient, the Muon update is written unscaled and the master
    moves by -lr * u ('Support Muon in BF16_Optimizer ...', PR
    description: Muon after reduction and global clipping)."""
    lay = wl.tiny_layout() if lay_name == "tiny" else mixed_layout()
    st = make_state(torch, lay, 61)
    before = st.numpy()
    gres = nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                       BETA, LR, method, 5, CLIP, mode, clip_mode="grad"))
    oa, om_, ow, r = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, 5, CLIP,
                                       ORACLE_MODE[mode], clip_mode="grad")
    ga, gm, gw = st.numpy()
    assert gres["applied"] == 1 and r["coef"] < 1.0
    assert abs(gres["global_norm"] - r["norm"]) <= 1e-6 * r["norm"]
    assert abs(gres["clip_coef"] - r["coef"]) <= 1e-6 * r["coef"]
    pad = wl.padding_mask(lay)
    for x0, x1 in zip(before, (ga, gm, gw)):
        assert np.array_equal(bits(x0)[pad], bits(x1)[pad]), "padding touched"
    mu, ax = muon_mask(lay), aux_mask(lay)
    # m' = beta m + coef g: a coefficient ulp moves m' by about |coef g| 2^-23,
    # however much the two terms cancel
    scale = np.abs(np.float32(BETA) * before[1][mu]) + np.abs(np.float32(r["coef"]) * before[0][mu])
    assert (np.abs(gm[mu] - om_[mu]) <= 1e-6 * scale).all(), "momentum"
    assert np.allclose(ga[ax], oa[ax], rtol=1e-6, atol=0), "auxiliary write-back"
    ug, uo = wl.unpack(lay, ga), wl.unpack(lay, oa)
    for k, spec in enumerate(lay.specs):
        if spec.use_muon:
            assert_close_update(ug[k], uo[k], mode, spec.name)
    w_expect = before[2].copy()
    w_expect[mu] = before[2][mu] - np.float32(LR) * ga[mu]
    assert np.array_equal(bits(gw), bits(w_expect)), "master = master - lr * u"
    assert nsg.device_error() == 0


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_inactive_gradient_clip_equals_update_clip(torch, method):
    """With the clip above every norm both orders have coefficient 1 and
    give bit-identical steps."""
    lay = mixed_layout()
    outs = []
    for cm in ("update", "grad"):
        st = make_state(torch, lay, 62)
        gres = nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params,
                                           lay.parts, BETA, LR, method, 5, 1e9, "bf16",
                                           clip_mode=cm))
        assert gres["clip_coef"] == 1.0
        outs.append(st.numpy())
    for a, b in zip(*outs):
        assert np.array_equal(bits(a), bits(b))


@pytest.mark.parametrize("clip_mode", ["update", "grad"])
@pytest.mark.parametrize("with_adam", [False, True])
def test_loss_scale_undo_bit_exact(torch, clip_mode, with_adam):
    """accum = 2^12 g with grad_scale 2^-12 reproduces the step on g bit for
    bit: the norm and the overflow check never see the loss scale ('Fix
    Muon optimizer under ZeRO CPU offload and bound gather buffers',
    loss-scaling commit)."""
    lay = mixed_layout()
    outs, res = [], []
    for scale, gs in ((1.0, 1.0), (4096.0, 2.0 ** -12)):
        st = make_state(torch, lay, 63, scale=scale, adam=with_adam)
        adam = adam_dict(st, 1) if with_adam else None
        res.append(nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params,
                                               lay.parts, BETA, LR, "gram", 5, CLIP, "bf16",
                                               clip_mode=clip_mode, grad_scale=gs, adam=adam)))
        o = list(st.numpy())
        if with_adam:
            o += [st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()]
        outs.append(o)
    assert res[0] == res[1]
    for a, b in zip(*outs):
        assert np.array_equal(bits(a), bits(b))


def test_grad_scale_overflow_skips(torch):
    """A finite accumulator that the grad_scale pushes past FP32's range is
    an overflow: the step is skipped and nothing is written."""
    lay = mixed_layout()
    st = make_state(torch, lay, 64, adam=True)
    k = next(i for i, s in enumerate(lay.specs) if not s.use_muon)
    off = int(lay.params["offset"][k])
    # the one storage element holding flat index `off`
    q = lay.parts
    j = int(np.searchsorted(q["flat_end"], off, side="right"))
    st.accum[int(q["storage_offset"][j]) + off - int(q["flat_begin"][j])] = 3e38
    before = list(st.numpy()) + [st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()]
    gres = nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                       BETA, LR, "gram", 5, CLIP, "bf16", grad_scale=4.0,
                                       adam=adam_dict(st, 1)))
    assert gres["applied"] == 0
    after = list(st.numpy()) + [st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()]
    for a, b in zip(before, after):
        assert np.array_equal(bits(a), bits(b))


@pytest.mark.parametrize("clip_mode", ["update", "grad"])
def test_aux_adam_three_steps_bit_exact(torch, clip_mode):
    """Fused Adam on the auxiliary groups over three steps (t = 1, 2, 3),
    clip off: exp_avg, exp_avg_sq and the auxiliary master are bit-exact
    against the oracle's Adam (Kingma & Ba), Muon's results are unchanged
    by it, and only auxiliary elements of the Adam buffers are written."""
    lay = mixed_layout()
    st = make_state(torch, lay, 65, adam=True)
    ref = make_state(torch, lay, 65)
    ea0 = st.exp_avg.cpu().numpy()
    eas0 = st.exp_avg_sq.cpu().numpy()
    ax = aux_mask(lay)
    for t in (1, 2, 3):
        before = st.numpy()
        if t > 1:
            # a fresh gradient each step, the same on both states
            g = wl.storage_with_sentinels(lay, wl.gaussian_grads(lay, 65, 10 + t))
            st.accum.copy_(to_dev(g, torch))
            ref.accum.copy_(to_dev(g, torch))
            before = st.numpy()
        nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "gram", 5,
                    0.0, "bf16", clip_mode=clip_mode, adam=adam_dict(st, t))
        nsg.step_ex(ref.accum, ref.momentum, ref.master, lay.params, lay.parts, BETA, LR, "gram",
                    5, 0.0, "bf16", clip_mode=clip_mode)
        oa, om_, ow, r = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, "gram", 5,
                                           0.0, "bf16", clip_mode=clip_mode,
                                           adam=dict(ADAM, step=t), exp_avg=ea0, exp_avg_sq=eas0)
        ga, gm, gw = st.numpy()
        ea, eas = st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()
        assert np.array_equal(bits(ea), bits(r["exp_avg_buf"])), f"exp_avg at t={t}"
        assert np.array_equal(bits(eas), bits(r["exp_avg_sq_buf"])), f"exp_avg_sq at t={t}"
        assert np.array_equal(bits(gw[ax]), bits(ow[ax])), f"auxiliary master at t={t}"
        assert np.array_equal(bits(ga[ax]), bits(oa[ax]))
        ra, rm, rw = ref.numpy()
        assert np.array_equal(bits(ga), bits(ra)) and np.array_equal(bits(gm), bits(rm))
        assert np.array_equal(bits(gw[~ax]), bits(rw[~ax])), "Adam touched a Muon master"
        ea0, eas0 = ea, eas
    assert nsg.device_error() == 0


def test_aux_adam_with_active_clip(torch):
    """Adam takes the clipped auxiliary gradient coef * g."""
    lay = mixed_layout()
    st = make_state(torch, lay, 66, adam=True)
    before = st.numpy()
    ea0, eas0 = st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()
    gres = nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                       BETA, LR, "standard", 5, CLIP, "bf16",
                                       adam=adam_dict(st, 4)))
    _, _, ow, r = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, "standard", 5, CLIP,
                                    "bf16", adam=dict(ADAM, step=4), exp_avg=ea0, exp_avg_sq=eas0)
    assert r["coef"] < 1.0 and abs(gres["clip_coef"] - r["coef"]) <= 1e-2 * r["coef"]
    ax = aux_mask(lay)
    # the clip coefficient comes from the Muon updates (BF16 operands): its
    # relative error bounds that of every Adam quantity to first order
    c_err = abs(gres["clip_coef"] - r["coef"]) / r["coef"] + 1e-6
    ea = st.exp_avg.cpu().numpy()
    assert np.allclose(ea[ax], r["exp_avg_buf"][ax], rtol=2 * c_err, atol=0)
    gw = st.master.cpu().numpy()
    # Adam's step m / sqrt(v) is scale-free: the master hardly moves with coef
    assert np.allclose(gw[ax], ow[ax], rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("storage,nparts", [("identity", 1), ("rank_major", 4), ("shuffled", 7)])
def test_options_partition_independence_bitwise(torch, storage, nparts):
    """Gradient clip, loss-scale undo and Adam keep the step bitwise
    independent of the partition table."""
    outs = []
    for lay in (mixed_layout(2), mixed_layout(nparts, storage, 9)):
        st = make_state(torch, lay, 67, scale=256.0, adam=True)
        nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "gram", 5,
                    CLIP, "bf16", clip_mode="grad", grad_scale=1 / 256, adam=adam_dict(st, 2))
        outs.append([wl.unpack(lay, x) for x in
                     list(st.numpy()) + [st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()]])
    for xa, xb in zip(*outs):
        for a, b in zip(xa, xb):
            assert np.array_equal(bits(a), bits(b))


def _buffers(st, adam):
    out = list(st.numpy())
    if adam:
        out += [st.exp_avg.cpu().numpy(), st.exp_avg_sq.cpu().numpy()]
    return out


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
@pytest.mark.parametrize("clip_mode", ["update", "grad"])
def test_bounded_workspace_bit_identical(torch, method, mode, clip_mode):
    """workspace_budget runs the Newton-Schulz blocks in waves over a shared
    workspace ('Run Muon once per optimizer step under ZeRO-3 ...', 'The
    change': bounded per-rank buffers; 'Fix Muon optimizer under ZeRO CPU
    offload and bound gather buffers': a byte cap on gathered parameters).
    Every budget -- one block per wave, a few blocks, all -- gives the
    unbounded step's bits, Adam state included."""
    lay = mixed_layout()
    outs, res = [], []
    for budget in (0, 1, 40_000, 200_000, 1 << 40):
        st = make_state(torch, lay, 68, adam=True)
        res.append(nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params,
                                               lay.parts, BETA, LR, method, 5, CLIP, mode,
                                               clip_mode=clip_mode, adam=adam_dict(st, 2),
                                               workspace_budget=budget)))
        outs.append(_buffers(st, True))
    for k in range(1, len(outs)):
        assert res[k] == res[0], k
        for a, b in zip(outs[0], outs[k]):
            assert np.array_equal(bits(a), bits(b)), k
    assert nsg.device_error() == 0


def test_bounded_workspace_gpt2_layers_and_memory(torch):
    """Two GPT-2-small layers, P=8, 16 MiB budget: bit-identical to the
    unbounded step, several waves, and the workspace stays within the budget
    (every block here fits it)."""
    lay = wl.gpt2_small_layout(layers=2)
    budget = 16 << 20
    outs = []
    for b in (0, budget):
        nsg.release_workspace()
        st = make_state(torch, lay, 69)
        nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "standard",
                    5, CLIP, "bf16", workspace_budget=b)
        outs.append(list(st.numpy()))
        ws = nsg.get_stats()["workspace_bytes"]
        if b:
            assert ws <= budget + 4096, ws
        else:
            assert ws > 3 * budget, ws
    for a, b in zip(*outs):
        assert np.array_equal(bits(a), bits(b))
    nsg.release_workspace()


def test_bounded_workspace_overflow_skips(torch):
    lay = mixed_layout()
    st = make_state(torch, lay, 70)
    st.accum[int(lay.params["offset"][1])] = float("nan")
    before = st.numpy()
    gres = nsg.read_result(nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                       BETA, LR, "gram", 5, CLIP, "bf16", workspace_budget=1))
    assert gres["applied"] == 0
    for a, b in zip(before, st.numpy()):
        assert np.array_equal(bits(a), bits(b))
