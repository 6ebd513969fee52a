"""The step's folded micro-batches (muon_step_ex's last_grad, and prev_grad
before it): the step accumulates the last one or two bf16 micro-batches
itself, in its first read of accum, with muon_accumulate's arithmetic.  accum, momentum, master and the device
result must therefore equal, bit for bit, muon_accumulate on that
micro-batch followed by the step; that sequence is itself checked against
the oracle by the parity tests.  Padding holds NaN sentinels and must come
out unchanged on both paths."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import GpuState, bf16_tensor, bits, micro_batch_grads

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def mixed_layout(nparts, storage):
    """Muon blocks in both orientations (one split into heads), aligned and
    ragged auxiliary groups: fast and element-wise tiles of the first pass."""
    return wl.build_layout(
        [[wl.ParamSpec("wq", 128, 192, 4), wl.ParamSpec("wt", 192, 128)],
         [wl.ParamSpec("ln", 1, 768, use_muon=False), wl.ParamSpec("emb", 40, 768, use_muon=False)],
         [wl.ParamSpec("odd", 7, 5, use_muon=False), wl.ParamSpec("w17", 17, 13)]], 128, nparts,
        storage, 7)


def misaligned(t, torch):
    """The same bf16 values at an address that is 8- but not 16-byte
    aligned (the step's 8-byte loads of folded micro-batches)."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)[4:]
    buf.copy_(t)
    assert buf.data_ptr() % 16 == 8
    return buf


ADAM = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=3)


def run(torch, lay, grads, gas, fold, method, mode, nan_last=False, misalign=False, adam=False,
        **opts):
    """accumulate the micro-batches (all, or all but the last `fold` of
    them, which the step folds in: 1 = last_grad, 2 = prev_grad and
    last_grad), then one step; returns the three storage buffers and the
    result (with `adam`: the auxiliary Adam step on fresh moments, which are
    returned after the master)."""
    m = [np.float32(0.01) * x for x in wl.gaussian_grads(lay, 11, 1, None, bf16=False)]
    w = wl.gaussian_grads(lay, 11, 2, None, bf16=False)
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.storage_with_sentinels(lay, z), wl.storage_with_sentinels(lay, m),
                  wl.storage_with_sentinels(lay, w))
    g = [list(x) for x in grads]
    if nan_last:
        g[-1][0] = g[-1][0].copy()
        g[-1][0].flat[3] = np.nan
    gb = [bf16_tensor(wl.bf16_storage_grad(lay, x), torch) for x in g]
    if misalign:
        gb = [misaligned(x, torch) for x in gb]
    fold = min(int(fold), gas)
    for mb in range(gas - fold):
        nsg.accumulate(st.accum, gb[mb], 1.0 / gas, overwrite=(mb == 0), params=lay.params,
                       parts=lay.parts)
    if fold:
        opts.update(last_grad=gb[-1], last_grad_scale=1.0 / gas, last_grad_overwrite=(gas == 1))
    if fold == 2:
        opts.update(prev_grad=gb[-2], prev_grad_scale=1.0 / gas, prev_grad_overwrite=(gas == 2))
    moments = []
    if adam:
        zero = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
        moments = [torch.from_numpy(wl.storage_with_sentinels(lay, zero)).cuda() for _ in range(2)]
        opts["adam"] = dict(ADAM, exp_avg=moments[0], exp_avg_sq=moments[1])
    res = nsg.step_ex(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, method, 5,
                      CLIP, mode, **opts)
    bufs = st.numpy()
    if adam:
        return tuple(bufs) + tuple(x.cpu().numpy() for x in moments), nsg.read_result(res)
    return bufs, nsg.read_result(res)


CASES = [
    # nparts, storage, gas, method, mode, options
    (3, "shuffled", 3, "standard", "bf16", {}),
    (2, "rank_major", 1, "gram", "fp32", {}),
    (3, "identity", 2, "standard", "bf16", {"clip_mode": "grad"}),
    (2, "shuffled", 2, "gram", "bf16", {"workspace_budget": 1}),
    (3, "identity", 4, "standard", "fp32", {"grad_scale": 0.5}),
    (2, "shuffled", 2, "standard", "bf16", {"adam": True}),
    (3, "rank_major", 2, "gram", "bf16", {"adam": True, "clip_mode": "grad"}),
]


@pytest.mark.parametrize("fold", [1, 2])
@pytest.mark.parametrize("nparts,storage,gas,method,mode,opts", CASES)
def test_folded_last_micro_batch_is_bit_identical(torch, nparts, storage, gas, method, mode, opts,
                                                  fold):
    lay = mixed_layout(nparts, storage)
    grads = micro_batch_grads(lay, 5, 0, gas, wl.loguniform_sigmas(lay, 5, 1e-3, 1e-1))
    b0, r0 = run(torch, lay, grads, gas, 0, method, mode, **dict(opts))
    b1, r1 = run(torch, lay, grads, gas, fold, method, mode, **dict(opts))
    assert r0["applied"] == 1 and r1 == r0
    for x, y in zip(b0, b1):   # accum, momentum, master (and the Adam moments)
        np.testing.assert_array_equal(bits(x), bits(y))
    pad = wl.padding_mask(lay)
    assert (bits(b1[0])[pad] == wl.NAN_SENTINEL_BITS).all()


@pytest.mark.parametrize("gas,fold,opts", [(3, 1, {}), (3, 2, {}), (2, 2, {}), (1, 1, {}),
                                           (2, 2, {"workspace_budget": 1}),
                                           (2, 2, {"clip_mode": "grad"})])
def test_folded_non_finite_micro_batch_skips_identically(torch, gas, fold, opts):
    """A skipped step leaves the accumulated gradient in accum, whether the
    first pass wrote it (gas 3) or the step writes it only on a skip (the
    folded micro-batches overwrite accum: gas 2 and 1; also in waves and
    with the gradient clipped before Muon)."""
    lay = mixed_layout(3, "shuffled")
    grads = micro_batch_grads(lay, 6, 0, gas)
    (a0, m0, w0), r0 = run(torch, lay, grads, gas, 0, "standard", "bf16", nan_last=True, **opts)
    (a1, m1, w1), r1 = run(torch, lay, grads, gas, fold, "standard", "bf16", nan_last=True, **opts)
    assert r0["applied"] == 0 and r1 == r0
    for x, y in ((a0, a1), (m0, m1), (w0, w1)):
        np.testing.assert_array_equal(bits(x), bits(y))


@pytest.mark.parametrize("gas,fold,misalign", [(4, 1, False), (4, 2, False), (2, 2, False),
                                               (2, 2, True), (1, 1, False)])
def test_folded_large_layout_matches(torch, gas, fold, misalign):
    """GPT-2-small-shaped blocks (one layer, P = 8): the fast paths over
    large tiles.  gas 4: the folded micro-batches add to accum (the first
    pass writes the gradient); gas 2 and 1: they overwrite it (every pass
    forms the gradient, 16-byte loads of 16-byte aligned micro-batches,
    8-byte loads of misaligned ones)."""
    lay = wl.build_layout([[wl.ParamSpec("q", 768, 768, 12), wl.ParamSpec("k", 768, 768, 12),
                            wl.ParamSpec("v", 768, 768), wl.ParamSpec("up", 3072, 768),
                            wl.ParamSpec("down", 768, 3072)]], 128, 8)
    grads = micro_batch_grads(lay, 8, 0, gas, wl.loguniform_sigmas(lay, 8, 1e-4, 1e-1))
    (a0, m0, w0), r0 = run(torch, lay, grads, gas, 0, "standard", "bf16")
    (a1, m1, w1), r1 = run(torch, lay, grads, gas, fold, "standard", "bf16", misalign=misalign)
    assert r0["applied"] == 1 and r1 == r0
    for x, y in ((a0, a1), (m0, m1), (w0, w1)):
        np.testing.assert_array_equal(bits(x), bits(y))


def test_folded_llama3_8b_step_matches_accumulate_then_step(torch):
    """The benchmark's configuration at full size (Llama-3-8B, 6.98G
    elements, P = 64, both bf16 micro-batches folded with overwrite, so
    every pass forms the gradient from them): accum, momentum and master
    after the step equal those of muon_accumulate twice followed by the
    step -- fingerprinted in 64M-element chunks (exact integer sums of the
    bit patterns) and bit for bit on six sampled matrices of both
    orientations."""
    lay = wl.llama3_8b_layout()
    seed = wl.CONFIG_SEED["llama"]
    n = lay.storage_size
    P, Q = lay.params, lay.parts
    g = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for mb in range(2):
        wl.llama_grad_into(lay, seed, mb, g[mb])
    state = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    sample = [1, 3, 5, 7 * 31 + 1, 7 * 31 + 4, 7 * 31 + 6]
    chunk = 1 << 26

    def run(fold):
        acc, mom, mst = state
        acc.zero_()
        mom.copy_(g[1]).mul_(0.1)
        mst.copy_(g[0])
        opts = None
        if fold:
            opts = nsg.step_options(prev_grad=g[0], prev_grad_scale=0.5, prev_grad_overwrite=True,
                                    last_grad=g[1], last_grad_scale=0.5)
        else:
            for mb in range(2):
                nsg.accumulate(acc, g[mb], 0.5, overwrite=(mb == 0), params=P, parts=Q)
        res = nsg.read_result(nsg.step(acc, mom, mst, P, Q, BETA, LR, "standard", 5, 0.0, "bf16",
                                       options=opts))
        prints = [torch.stack([t.view(torch.int32)[i:i + chunk].sum(dtype=torch.int64)
                               for i in range(0, n, chunk)]).cpu().numpy() for t in state]
        mats = []
        for k in sample:
            off, s = int(P["offset"][k]), lay.specs[k]
            mats.append([t[off:off + s.numel].cpu().numpy() for t in state])
        return res, prints, mats

    r0, p0, m0 = run(False)
    r1, p1, m1 = run(True)
    assert r0["applied"] == 1 and r1 == r0
    for a, b in zip(p0, p1):
        np.testing.assert_array_equal(a, b)
    for x, y in zip(m0, m1):
        for a, b in zip(x, y):
            np.testing.assert_array_equal(bits(a), bits(b))
    del g, state
    nsg.release_workspace()
    torch.cuda.empty_cache()
    assert nsg.device_error() == 0
