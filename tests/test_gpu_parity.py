"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Each test builds seeded inputs with ``workloads``, runs the library on the
GPU and the oracle on the CPU from the same inputs, and compares with the
rules in ``harness``: bit-exact for accumulation, momentum, ownership,
padding and skips; per-matrix tolerances for the Newton-Schulz update."""

import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import oracle.bf16 as obf
import oracle.muon as om
import oracle.newton_schulz as ons
import workloads as wl
from harness import (ORACLE_MODE, GpuState, assert_close_update, bf16_tensor, bits,
                     micro_batch_grads, relf, to_dev)

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05
BAND_LO, BAND_HI = 0.6818, 1.2024


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def oracle_accumulate(acc, layout, grads, gas):
    """Oracle S1 on storage buffers: parameter elements only."""
    pad = wl.padding_mask(layout)
    out = acc.copy()
    for mb, g in enumerate(grads):
        gv = obf.bits_to_f32(wl.bf16_storage_grad(layout, g))
        out[~pad] = om.accumulate(out[~pad], gv[~pad], 1.0 / gas, overwrite=(mb == 0))
    return out


def gpu_accumulate(st, layout, grads, gas, torch):
    for mb, g in enumerate(grads):
        gb = bf16_tensor(wl.bf16_storage_grad(layout, g), torch)
        nsg.accumulate(st.accum, gb, 1.0 / gas, overwrite=(mb == 0), params=layout.params,
                       parts=layout.parts)


def check_step(layout, before, after, ores, gres, mode, pad, sample=None):
    """Compare one step: momentum bit-exact, update per matrix, master
    bit-exact given the update, padding untouched."""
    a0, m0, w0 = before
    ga, gm, gw = after
    oa, om_, ow = ores[:3]
    r = ores[3]
    assert gres["applied"] == 1 == r["applied"]
    assert np.array_equal(bits(gm), bits(om_)), "momentum differs"
    for x0, x1 in [(a0, ga), (m0, gm), (w0, gw)]:
        assert np.array_equal(bits(x0)[pad], bits(x1)[pad]), "padding touched"
    tol = 1e-2 if mode == "bf16" else 1e-5
    assert abs(gres["global_norm"] - r["norm"]) <= tol * r["norm"] + 1e-30
    assert abs(gres["clip_coef"] - r["coef"]) <= tol * r["coef"] + 1e-30
    ug, uo = wl.unpack(layout, ga), wl.unpack(layout, oa)
    for k, spec in enumerate(layout.specs):
        if sample is not None and k not in sample:
            continue
        if spec.use_muon:
            assert_close_update(ug[k] / gres["clip_coef"], uo[k] / r["coef"], mode, spec.name)
        else:
            assert np.allclose(ug[k], uo[k], rtol=tol, atol=0), spec.name
    # master = master - lr * update, in float32, exactly from the GPU's own update
    w_expect = w0.copy()
    cov = wl.pack(layout, [np.full((s.rows, s.cols), 1 if s.use_muon else 0, np.int8)
                           for s in layout.specs], np.int8, 0).astype(bool)
    w_expect[cov] = w0[cov] - np.float32(LR) * ga[cov]
    assert np.array_equal(bits(gw), bits(w_expect)), "master write differs"


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_tiny_config_three_steps(torch, method, mode):
    """17x13 and 9x17 Muon matrices plus an 8x5 auxiliary group, two
    partitions cutting both matrices, gas=3, clip 0.05, three steps
    ('Support Muon in BF16_Optimizer ...', validation table, eager E2E)."""
    lay = wl.tiny_layout()
    seed = wl.CONFIG_SEED["tiny"]
    rng = wl.rng_for(seed, 777)
    w0 = [(0.02 * rng.standard_normal((s.rows, s.cols))).astype(np.float32) for s in lay.specs]
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.storage_with_sentinels(lay, z), wl.storage_with_sentinels(lay, z),
                  wl.storage_with_sentinels(lay, w0))
    pad = wl.padding_mask(lay)
    for step in range(3):
        grads = micro_batch_grads(lay, seed, step, 3)
        a_pre = st.accum.cpu().numpy()
        gpu_accumulate(st, lay, grads, 3, torch)
        before = st.numpy()
        assert np.array_equal(bits(before[0]), bits(oracle_accumulate(a_pre, lay, grads, 3)))
        res = nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR,
                       method, 5, CLIP, mode)
        gres = nsg.read_result(res)
        assert gres["ns_calls"] == 2
        ores = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, 5, CLIP,
                                 ORACLE_MODE[mode])
        check_step(lay, before, st.numpy(), ores, gres, mode, pad)
    assert nsg.device_error() == 0


@pytest.mark.parametrize("storage,nparts", [("identity", 1), ("identity", 8),
                                            ("rank_major", 2), ("shuffled", 8)])
def test_partition_independence_bitwise(torch, storage, nparts):
    """Results do not depend on where partition boundaries fall or where
    partitions are stored: bit-identical to the P=2 identity layout."""
    results = []
    for lay in [wl.gpt2_small_layout(layers=1, nparts=2),
                wl.gpt2_small_layout(layers=1, nparts=nparts, storage=storage, seed=5)]:
        seed = 31
        mats_g = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-4, 1e-1))
        mats_m = wl.gaussian_grads(lay, seed, 1, None, bf16=False)
        mats_w = wl.gaussian_grads(lay, seed, 2, None, bf16=False)
        st = GpuState(torch, wl.storage_with_sentinels(lay, mats_g),
                      wl.storage_with_sentinels(lay, mats_m), wl.storage_with_sentinels(lay, mats_w))
        pad = wl.padding_mask(lay)
        before = st.numpy()
        nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "standard", 5,
                 CLIP, "bf16")
        after = st.numpy()
        for x0, x1 in zip(before, after):
            assert np.array_equal(bits(x0)[pad], bits(x1)[pad])
        results.append([wl.unpack(lay, x) for x in after])
    for xa, xb in zip(results[0], results[1]):
        for a, b in zip(xa, xb):
            assert np.array_equal(bits(a), bits(b))


def test_overflow_skips_and_leaves_state_untouched(torch):
    lay = wl.tiny_layout()
    mats = wl.gaussian_grads(lay, 5, 0)
    mats[1] = mats[1].copy()
    mats[1][2, 3] = np.inf
    m = wl.gaussian_grads(lay, 5, 1, None, bf16=False)
    st = GpuState(torch, wl.storage_with_sentinels(lay, mats), wl.storage_with_sentinels(lay, m),
                  wl.storage_with_sentinels(lay, m))
    before = st.numpy()
    gres = nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                    BETA, LR, "gram", 5, CLIP, "bf16"))
    assert gres["applied"] == 0 and gres["ns_calls"] == 0
    for x0, x1 in zip(before, st.numpy()):
        assert np.array_equal(bits(x0), bits(x1))
    # NaN sentinels in padding alone do not skip the step
    mats[1][2, 3] = 0.0
    st = GpuState(torch, wl.storage_with_sentinels(lay, mats), wl.storage_with_sentinels(lay, m),
                  wl.storage_with_sentinels(lay, m))
    assert nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                    BETA, LR, "gram", 5, CLIP, "bf16"))["applied"] == 1


def test_ns_once_per_matrix_per_step(torch):
    """2 matrices, 2 steps, gas=4: 4 Newton-Schulz calls ('Run Muon once per
    optimizer step under ZeRO-3 ...', 'The problem' table)."""
    lay = wl.build_layout([[wl.ParamSpec("a", 6, 10), wl.ParamSpec("b", 10, 6)]], 16, 2)
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.pack(lay, z), wl.pack(lay, z), wl.pack(lay, z))
    total = 0
    for step in range(2):
        gpu_accumulate(st, lay, micro_batch_grads(lay, 9, step, 4), 4, torch)
        total += nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                          BETA, LR, "gram", 5, 0.0, "bf16"))["ns_calls"]
        assert nsg.get_stats()["ns_calls_last_step"] == 2
    assert total == 4


def test_gas_equivalence_bitwise(torch):
    """gas=1 with the mean gradient and gas=4 with four exact parts give
    bit-identical steps ('Run Muon once per optimizer step ...', 'The
    problem': the same samples in one or four micro-batches)."""
    lay = wl.gpt2_small_layout(layers=1, nparts=4)
    rng = wl.rng_for(41)
    parts4 = [[(rng.integers(-64, 65, (s.rows, s.cols)) / 64.0).astype(np.float32)
               for s in lay.specs] for _ in range(4)]
    mean = [sum(p[k] for p in parts4) / 4 for k in range(len(lay.specs))]
    outs = []
    for grads, gas in [([mean], 1), (parts4, 4)]:
        z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
        st = GpuState(torch, wl.pack(lay, z), wl.pack(lay, z), wl.pack(lay, z))
        gpu_accumulate(st, lay, grads, gas, torch)
        nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "standard", 5,
                 CLIP, "bf16")
        outs.append(st.numpy())
    for a, b in zip(*outs):
        assert np.array_equal(bits(a), bits(b))


NS_SHAPES = [(77, 300), (300, 77), (1000, 1500), (1024, 1024), (13, 17)]


@pytest.mark.parametrize("shape", NS_SHAPES)
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_newton_schulz_entry(torch, shape, method, mode):
    G = wl.rng_for(51, *shape).standard_normal(shape).astype(np.float32)
    if mode == "bf16":
        G = wl.to_bf16_values(G)
        X = to_dev(G, torch, torch.bfloat16)
    else:
        X = to_dev(G, torch)
    Y = nsg.newton_schulz(X, ns_method=method, ns_steps=5, operand_mode=mode)
    want = ons.newton_schulz(G, method, 5, ORACLE_MODE[mode])
    assert_close_update(Y.float().cpu().numpy(), want, mode, f"{shape} {method} {mode}")


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_tensor_core_path_matches_cuda_core_path(torch, method, mode):
    """The tensor-core products (BF16 operands, or FP32 through split-3
    planes) against the CUDA-core products on one matrix, both by the
    mode's rule, and both against the oracle."""
    G = wl.rng_for(52).standard_normal((640, 1100)).astype(np.float32)
    if mode == "bf16":
        G = wl.to_bf16_values(G)
        X = to_dev(G, torch, torch.bfloat16)
    else:
        X = to_dev(G, torch)
    outs = []
    for path in ("default", "simt"):
        with nsg.testing(gemm=path):
            outs.append(nsg.newton_schulz(X, ns_method=method, operand_mode=mode)
                        .float().cpu().numpy())
    assert_close_update(outs[0], outs[1], mode, f"tensor vs cuda cores {method} {mode}")
    want = ons.newton_schulz(G, method, 5, ORACLE_MODE[mode])
    for o in outs:
        assert_close_update(o, want, mode, f"{method} {mode} vs oracle")


@pytest.mark.parametrize("method,mode", [("standard", "bf16"), ("gram", "bf16"),
                                         ("standard", "fp32"), ("gram", "fp32")])
def test_gpt2_small_config(torch, method, mode):
    """GPT-2-small shapes: 12 layers of Q, K (12 heads), V, O 768x768,
    up 3072x768, down 768x3072; P=8, 128 alignment; gas=4, bf16 grads with
    per-matrix sigma log-uniform in [1e-4, 1e-1]; one step in each method
    and operand mode.  Accumulation and momentum bit-exact everywhere; every
    one of the 72 matrices against the oracle by the mode's rule; every
    block's update in the quintic's band."""
    lay = wl.gpt2_small_layout()
    seed = wl.CONFIG_SEED["gpt2"]
    sig = wl.loguniform_sigmas(lay, seed, 1e-4, 1e-1)
    grads = micro_batch_grads(lay, seed, 0, 4, sig)
    m0 = [0.1 * s for s in wl.gaussian_grads(lay, seed, 100, sig, bf16=False)]
    w0 = wl.gaussian_grads(lay, seed, 101, None, bf16=False)
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.pack(lay, z), wl.pack(lay, m0), wl.pack(lay, w0))
    gpu_accumulate(st, lay, grads, 4, torch)
    before = st.numpy()
    assert np.array_equal(bits(before[0]), bits(oracle_accumulate(wl.pack(lay, z), lay, grads, 4)))
    gres = nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                    BETA, LR, method, 5, CLIP, mode))
    assert gres["applied"] == 1 and gres["ns_calls"] == 12 * 28
    ga, gm, gw = st.numpy()
    g_un, m_un, u_un = wl.unpack(lay, before[0]), wl.unpack(lay, before[1]), wl.unpack(lay, ga)
    mom_un = wl.unpack(lay, gm)
    for k, spec in enumerate(lay.specs):
        want_m = om.momentum_update(m_un[k], g_un[k], BETA)
        assert np.array_equal(bits(mom_un[k]), bits(want_m)), spec.name
        u = u_un[k] / gres["clip_coef"]
        assert np.all(np.isfinite(u))
        h = spec.num_heads if spec.num_heads > 1 else 1
        br = spec.rows // h
        for b in range(h):
            blk = u[b * br:(b + 1) * br].astype(np.float64)
            mm = min(blk.shape)
            sq = float(np.sum(blk * blk))
            assert mm * BAND_LO ** 2 * 0.98 <= sq <= mm * BAND_HI ** 2 * 1.02, (spec.name, b, sq / mm)
    for k, spec in enumerate(lay.specs):         # all 72 matrices
        _, u_or = om.muon_update(g_un[k], m_un[k], BETA, method, 5, spec.num_heads,
                                 ORACLE_MODE[mode])
        assert_close_update(u_un[k] / gres["clip_coef"], u_or, mode, f"{spec.name} {method} {mode}")


@pytest.mark.parametrize("nparts", [1, 8])
def test_ragged_small_matrices_gram(torch, nparts):
    """8192 matrices, rows from {32..256}, cols from {128..1024}, half tall;
    fp32 grads N(0,1) x 10^U(-5,0) written straight into accum; one gram
    step.  64 sampled matrices against the oracle, all in the band.  P = 1
    is the plain reading of the config; P = 8 puts partition boundaries
    through the packed small matrices of both orientations."""
    seed = wl.CONFIG_SEED["ragged"]
    lay = wl.ragged_layout(8192, nparts=nparts, seed=seed)
    rng = wl.rng_for(seed, 1)
    scales = 10.0 ** rng.uniform(-5, 0, len(lay.specs))
    mats = [(wl.rng_for(seed, 2, i).standard_normal((s.rows, s.cols)) * scales[i]).astype(np.float32)
            for i, s in enumerate(lay.specs)]
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    st = GpuState(torch, wl.pack(lay, mats), wl.pack(lay, z), wl.pack(lay, z))
    gres = nsg.read_result(nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts,
                                    BETA, LR, "gram", 5, 0.0, "bf16"))
    assert gres["applied"] == 1 and gres["ns_calls"] == 8192 and gres["clip_coef"] == 1.0
    u_un = wl.unpack(lay, st.accum.cpu().numpy())
    for k, spec in enumerate(lay.specs):
        blk = u_un[k].astype(np.float64)
        sq = float(np.sum(blk * blk))
        mm = min(blk.shape)
        assert mm * BAND_LO ** 2 * 0.98 <= sq <= mm * BAND_HI ** 2 * 1.02, (k, sq / mm)
    for k in wl.rng_for(seed, 3).choice(len(lay.specs), 64, replace=False):
        _, u_or = om.muon_update(mats[k], z[k], BETA, "gram", 5, 0, "bf16")
        assert_close_update(u_un[k], u_or, "bf16", lay.specs[k].name)


def test_llama3_8b_config_sampled(torch):
    """Llama-3-8B shapes at full size (6.98G elements, P=64, gas=2, standard
    NS): every block's update in the quintic band (checked on the device);
    sampled Gaussian matrices against the BF16 oracle; a sampled low-rank
    matrix by the declared rule (top-8 subspace within 1e-2, sigma_max
    within the band) and, in FP32 mode, against the exact oracle at
    atol 1e-4 / rtol 1e-3."""
    lay = wl.llama3_8b_layout()
    seed = wl.CONFIG_SEED["llama"]
    n = lay.storage_size
    acc = torch.zeros(n, dtype=torch.float32, device="cuda")
    mom = torch.zeros(n, dtype=torch.float32, device="cuda")
    mst = torch.zeros(n, dtype=torch.float32, device="cuda")
    grad = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    # k (1024x4096), o (4096^2) and up (14336x4096) of layer 0; k, v and
    # down (4096x14336) of layer 31
    sample = [1, 3, 5, 7 * 31 + 1, 7 * 31 + 2, 7 * 31 + 6]
    g_host = {k: [] for k in sample}
    for mb in range(2):
        wl.llama_grad_into(lay, seed, mb, grad)
        for k in sample:
            off, s = int(lay.params["offset"][k]), lay.specs[k]
            g_host[k].append(grad[off:off + s.numel].float().cpu().numpy().reshape(s.rows, s.cols))
        nsg.accumulate(acc, grad, 0.5, overwrite=(mb == 0), params=lay.params, parts=lay.parts)
    del grad
    res = nsg.read_result(nsg.step(acc, mom, mst, lay.params, lay.parts, BETA, LR, "standard", 5,
                                   0.0, "bf16"))
    assert res["applied"] == 1 and res["ns_calls"] == 224 and res["clip_coef"] == 1.0
    # band check of every block on the device: Gaussian blocks have all m
    # singular values in the band; rank-8-plus-1e-3-noise blocks have 8 in
    # the band and noise directions (normalised ~1e-5, amplified ~a^5 ~ 485)
    # that add well under 1 to the sum of squares
    for k, spec in enumerate(lay.specs):
        off = int(lay.params["offset"][k])
        u = acc[off:off + spec.numel].double()
        sq = float((u * u).sum())
        r = min(spec.rows, spec.cols) if k % 2 == 1 else 8
        extra = 0.0 if k % 2 == 1 else 1.0
        assert r * BAND_LO ** 2 * 0.98 <= sq <= r * BAND_HI ** 2 * 1.02 + extra, (spec.name, sq / r)
    for k in sample:
        spec = lay.specs[k]
        off = int(lay.params["offset"][k])
        g = om.accumulate(om.accumulate(None, g_host[k][0], 0.5, True), g_host[k][1], 0.5)
        m_gpu = mom[off:off + spec.numel].cpu().numpy().reshape(spec.rows, spec.cols)
        assert np.array_equal(bits(m_gpu), bits(om.momentum_update(np.zeros_like(g), g, BETA)))
        u_gpu = acc[off:off + spec.numel].cpu().numpy().reshape(spec.rows, spec.cols)
        u_or = ons.newton_schulz(m_gpu, "standard", 5, "bf16")
        if k % 2 == 1:            # Gaussian
            assert_close_update(u_gpu, u_or, "bf16", spec.name)
        else:                     # low-rank + noise: declared rule in BF16 mode
            U = np.linalg.svd(m_gpu.astype(np.float64), full_matrices=False)[0][:, :8]
            proj = lambda x: U @ (U.T @ np.asarray(x, np.float64))
            assert relf(proj(u_gpu), proj(u_or)) <= 1e-2, spec.name
            assert np.linalg.norm(u_gpu.astype(np.float64), 2) <= BAND_HI * (1 + 1e-2)
            # and at the strict tolerance in FP32 mode
            y32 = nsg.newton_schulz(torch.from_numpy(m_gpu).cuda(), ns_method="standard",
                                    operand_mode="fp32").cpu().numpy()
            assert_close_update(y32, ons.newton_schulz(m_gpu, "standard", 5, "exact"), "fp32",
                                spec.name + " fp32")
    del acc, mom, mst
    nsg.release_workspace()
    torch.cuda.empty_cache()
    assert nsg.device_error() == 0


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_stacked_head_blocks_match_separate_blocks(torch, method, mode):
    """Consecutive equal head blocks (GPT-2 Q/K: 12 blocks of 64 x 768) run
    stacked into block-diagonal problems of up to 256 rows; the step must
    agree with one problem per block (stacking off) within the operand
    mode's rule, and both with the oracle on a sampled block."""
    lay = wl.gpt2_small_layout(layers=1, nparts=2)
    seed = 77
    g = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-3, 1e-1))
    m = wl.gaussian_grads(lay, seed, 1, None, bf16=False)
    outs = []
    for stack in (1, 0):
        with nsg.testing(stack=stack):
            st = GpuState(torch, wl.pack(lay, g), wl.pack(lay, m), wl.pack(lay, m))
            before = st.numpy()
            nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, method, 5,
                     0.0, mode)
            outs.append(wl.unpack(lay, st.accum.cpu().numpy()))
    for k, spec in enumerate(lay.specs):
        assert_close_update(outs[0][k], outs[1][k], mode, f"stacked vs separate {spec.name}")
    res = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, 5, 0.0,
                            ORACLE_MODE[mode])
    want = wl.unpack(lay, res[0])
    assert_close_update(outs[0][0], want[0], mode, "stacked Q vs oracle")


@pytest.mark.parametrize("knobs", [{"flow": 0}, {"flow_lag": 1}, {"flow_lag": 1000},
                                   {"flow_waves": 3, "flow_lag": 1000}, {"raster": 1}])
def test_pair_dataflow_schedule_is_bitwise_neutral(torch, knobs):
    """The SM-pair kernel's task order and dependency counters change only
    when tiles run, never what they compute: one launch per product, the
    tightest wavefront, product-major order and grouped waves all give the
    default schedule's bits.  A dependency released too early would read a
    half-written operand and differ."""
    lay = wl.gpt2_small_layout(layers=2, nparts=4)
    seed = 78
    g = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-3, 1e-1))
    m = wl.gaussian_grads(lay, seed, 1, None, bf16=False)
    outs = []
    for e in ({}, knobs):
        with nsg.testing(**e):
            st = GpuState(torch, wl.pack(lay, g), wl.pack(lay, m), wl.pack(lay, m))
            nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, "standard",
                     5, CLIP, "bf16")
            outs.append(st.numpy())
    for a, b in zip(*outs):
        assert np.array_equal(bits(a), bits(b))
    assert nsg.device_error() == 0


def test_pair_tile_raster_is_bitwise_neutral(torch):
    """Column-grouped tile order (the default for products with an MN-major
    B and 128+ tiles: here 8 x 32 tiles of X' = B X) against row-major order:
    the same tiles, the same bits."""
    G = wl.to_bf16_values(wl.rng_for(58).standard_normal((2048, 8192)).astype(np.float32))
    X = to_dev(G, torch, torch.bfloat16)
    outs = []
    for raster in (0, 1):
        with nsg.testing(raster=raster):
            outs.append(nsg.newton_schulz(X, ns_method="standard", operand_mode="bf16")
                        .float().cpu().numpy())
    assert np.array_equal(bits(outs[0]), bits(outs[1]))
    assert nsg.device_error() == 0


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_pair_kernel_matches_single_sm_kernel(torch, method):
    """BF16 products on SM pairs (256x256 tiles, cta_group::2) against the
    single-SM kernel (128x256 tiles, the "tc1" cross-check) on one GPT-2 layer, both
    by the BF16 rule, and both against the oracle on a sampled block."""
    lay = wl.gpt2_small_layout(layers=1, nparts=2)
    seed = 79
    g = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-3, 1e-1))
    m = wl.gaussian_grads(lay, seed, 1, None, bf16=False)
    outs = []
    for path in ("default", "tc1"):
        with nsg.testing(gemm=path):
            st = GpuState(torch, wl.pack(lay, g), wl.pack(lay, m), wl.pack(lay, m))
            before = st.numpy()
            nsg.step(st.accum, st.momentum, st.master, lay.params, lay.parts, BETA, LR, method, 5,
                     0.0, "bf16")
            outs.append(wl.unpack(lay, st.accum.cpu().numpy()))
    for k, spec in enumerate(lay.specs):
        assert_close_update(outs[0][k], outs[1][k], "bf16", f"pairs vs single SM {spec.name}")
    res = om.muon_step_flat(*before, lay.params, lay.parts, BETA, LR, method, 5, 0.0, "bf16")
    want = wl.unpack(lay, res[0])
    for o in outs:
        assert_close_update(o[4], want[4], "bf16", "MLP-up vs oracle")
