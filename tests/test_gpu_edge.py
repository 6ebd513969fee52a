"""Degenerate inputs of the step, against the oracle: one-row, one-column
and 1x1 Muon matrices (m = 1: a single singular value), a Muon matrix whose
gradient and momentum are zero (X0 = 0 / (0 + 1e-7) = 0, so its update is
exactly zero while the others' are not), a table with only auxiliary
parameters (no Newton-Schulz at all), and an empty table."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import oracle.muon as om
import workloads as wl
from harness import ORACLE_MODE, GpuState, bits, micro_batch_grads
from test_gpu_parity import check_step, gpu_accumulate

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def run(torch, lay, method, mode, zero=()):
    seed = 41
    grads = micro_batch_grads(lay, seed, 0, 2)
    for mb in range(2):
        grads[mb] = [np.zeros_like(g) if s.name in zero else g for g, s in zip(grads[mb], lay.specs)]
    m0 = [np.zeros((s.rows, s.cols), np.float32) if s.name in zero else np.float32(0.01) * x
          for s, x in zip(lay.specs, wl.gaussian_grads(lay, seed, 5, None, bf16=False))]
    w0 = wl.gaussian_grads(lay, seed, 6, None, bf16=False)
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.storage_with_sentinels(lay, z), wl.storage_with_sentinels(lay, m0),
                  wl.storage_with_sentinels(lay, w0))
    gpu_accumulate(st, lay, grads, 2, torch)
    before = st.numpy()
    gres = nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA,
                                    LR, method, 5, CLIP, mode))
    ores = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, 5, CLIP,
                             ORACLE_MODE[mode])
    assert nsg.device_error() == 0
    return before, st.numpy(), ores, gres


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_degenerate_shapes_and_a_zero_matrix(torch, method, mode):
    lay = wl.build_layout(
        [[wl.ParamSpec("row", 1, 64), wl.ParamSpec("col", 64, 1), wl.ParamSpec("one", 1, 1)],
         [wl.ParamSpec("zero", 32, 48), wl.ParamSpec("w", 40, 72),
          wl.ParamSpec("aux", 3, 7, use_muon=False)]], 16, 3)
    before, after, ores, gres = run(torch, lay, method, mode, zero=("zero",))
    assert gres["ns_calls"] == 5
    names = [s.name for s in lay.specs]
    k_zero = names.index("zero")
    check_step(lay, before, after, ores, gres, mode, wl.padding_mask(lay),
               sample=[k for k in range(len(names)) if k != k_zero])
    # the zero matrix: update exactly zero in accum, master and momentum unchanged
    ug, mg, wg = (wl.unpack(lay, x)[k_zero] for x in after)
    w_in = wl.unpack(lay, before[2])[k_zero]
    assert not ug.any() and not mg.any()
    assert np.array_equal(bits(wg), bits(w_in))


def test_auxiliary_only_table(torch):
    lay = wl.build_layout([[wl.ParamSpec("ln", 1, 768, use_muon=False),
                            wl.ParamSpec("emb", 40, 96, use_muon=False)]], 128, 2)
    before, after, ores, gres = run(torch, lay, "gram", "bf16")
    assert gres["ns_calls"] == 0 and gres["applied"] == 1
    pad = wl.padding_mask(lay)
    # no Newton-Schulz: norm over the gradients, accum = coef g, master untouched
    assert abs(gres["global_norm"] - ores[3]["norm"]) <= 1e-5 * ores[3]["norm"]
    assert abs(gres["clip_coef"] - ores[3]["coef"]) <= 1e-5 * ores[3]["coef"]
    assert np.allclose(after[0][~pad], ores[0][~pad], rtol=1e-5, atol=0)
    assert np.array_equal(bits(after[2]), bits(before[2]))
    assert np.array_equal(bits(after[1]), bits(before[1]))


def test_empty_table(torch):
    acc, mom, mst = (torch.zeros(16, dtype=torch.float32, device="cuda") for _ in range(3))
    res = nsg.step(acc, mom, mst, [], [], BETA, LR, "gram", 5, CLIP, "bf16")
    r = nsg.read_result(res)
    assert r["applied"] == 1 and r["ns_calls"] == 0
    assert r["global_norm"] == 0.0 and r["clip_coef"] == 1.0
    assert not acc.any() and not mom.any() and not mst.any()


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_tall_head_blocks(torch, method, mode):
    """Per-head splits whose blocks are taller than wide, so every head block
    is transposed into its canonical orientation on its own (1536 x 64 in 4
    heads of 384 x 64; 96 x 32 in 2 heads of 48 x 32), beside a wide
    head-split matrix; partitions cut through the blocks."""
    lay = wl.build_layout(
        [[wl.ParamSpec("tall4", 1536, 64, 4), wl.ParamSpec("tall2", 96, 32, 2),
          wl.ParamSpec("wide3", 96, 320, 3)]], 32, 3)
    before, after, ores, gres = run(torch, lay, method, mode)
    assert gres["ns_calls"] == 4 + 2 + 3
    check_step(lay, before, after, ores, gres, mode, wl.padding_mask(lay))


@pytest.mark.parametrize("steps", [1, 2, 7])
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_other_step_counts(torch, steps, method, mode):
    """ns_steps other than 5, through the step and the NS entry, against the
    oracle with the same count."""
    from oracle import newton_schulz as ons
    from harness import assert_close_update, to_dev
    lay = wl.tiny_layout()
    seed = 43
    grads = micro_batch_grads(lay, seed, 0, 1)
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.storage_with_sentinels(lay, z), wl.storage_with_sentinels(lay, z),
                  wl.storage_with_sentinels(lay, z))
    gpu_accumulate(st, lay, grads, 1, torch)
    before = st.numpy()
    gres = nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA,
                                    LR, method, steps, CLIP, mode))
    ores = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, steps, CLIP,
                             ORACLE_MODE[mode])
    check_step(lay, before, st.numpy(), ores, gres, mode, wl.padding_mask(lay))
    G = wl.rng_for(seed, 300, 77).standard_normal((300, 77)).astype(np.float32)
    if mode == "bf16":
        G = wl.to_bf16_values(G)
    X = to_dev(G, torch, torch.bfloat16 if mode == "bf16" else None)
    Y = nsg.newton_schulz(X, ns_method=method, ns_steps=steps, operand_mode=mode)
    assert_close_update(Y.float().cpu().numpy(), ons.newton_schulz(G, method, steps, ORACLE_MODE[mode]),
                        mode, f"NS entry {method} {mode} steps={steps}")
    assert nsg.device_error() == 0
