"""The bounds-checking build (MUON_DEBUG), standing in for a memory
sanitizer: its streaming kernels check, before a block touches memory,
that the block's tile stays inside the storage extent the partition table
describes and inside its owner's workspace region, and record error 16
instead of an out-of-range access.

In a fresh process that loads the debug library, a set of steps over the
layouts with the most varied tiles (partitions cutting matrices, shuffled
and rank-major storage, head blocks, transposed blocks, ragged auxiliary
groups, waves of a bounded workspace) must report no error, and their
accum, momentum and master must equal the release library's bit for bit
(the checks change no arithmetic).  A planted mismatch -- the checks told
that the storage is 64 elements shorter than the partitions say -- must be
reported as error 16, with no fault (muon_accumulate and
muon_accumulate_n).  The cases bring their two micro-batches to the step by
two muon_accumulate calls, by one muon_accumulate_n, or folded into the
step (the gradient formed by every pass, accum written by the write-back)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import bits

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def layouts():
    mixed = wl.build_layout(
        [[wl.ParamSpec("wq", 128, 192, 4), wl.ParamSpec("wt", 192, 128)],
         [wl.ParamSpec("ln", 1, 768, use_muon=False), wl.ParamSpec("emb", 40, 768, use_muon=False)],
         [wl.ParamSpec("odd", 7, 5, use_muon=False), wl.ParamSpec("w17", 17, 13)]], 128, 3,
        "shuffled", 7)
    # the last field: how the two micro-batches reach the step -- two
    # muon_accumulate calls, one muon_accumulate_n, or folded into the step
    return [("tiny", wl.tiny_layout(), "gram", "bf16", {}, "each"),
            ("tiny rank-major", wl.tiny_layout(nparts=2, storage="rank_major"), "standard", "fp32", {},
             "n"),
            ("gpt2 layer shuffled", wl.gpt2_small_layout(layers=1, nparts=8, storage="shuffled"),
             "standard", "bf16", {}, "fold"),
            ("mixed waves", mixed, "gram", "bf16", {"workspace_budget": 1}, "n"),
            ("mixed folded", mixed, "standard", "bf16", {}, "fold"),
            ("ragged", wl.ragged_layout(64, nparts=8), "gram", "fp32", {}, "each")]


def run_cases(torch):
    """Every layout: two micro-batches and one step; returns the buffers."""
    out = {}
    for name, lay, method, mode, opts, how in layouts():
        g = [wl.bf16_storage_grad(lay, wl.gaussian_grads(lay, 21, mb)) for mb in range(2)]
        m0 = [0.1 * x for x in wl.gaussian_grads(lay, 21, 5, None, bf16=False)]
        w0 = wl.gaussian_grads(lay, 21, 6, None, bf16=False)
        acc = torch.from_numpy(wl.storage_with_sentinels(
            lay, [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs])).cuda()
        mom = torch.from_numpy(wl.storage_with_sentinels(lay, m0)).cuda()
        mst = torch.from_numpy(wl.storage_with_sentinels(lay, w0)).cuda()
        gb = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in g]
        if how == "each":
            for mb in range(2):
                nsg.accumulate(acc, gb[mb], 0.5, overwrite=(mb == 0), params=lay.params,
                               parts=lay.parts)
        elif how == "n":
            nsg.accumulate_n(acc, gb, 0.5, overwrite=True, params=lay.params, parts=lay.parts)
        else:
            opts = dict(opts, prev_grad=gb[0], prev_grad_scale=0.5, prev_grad_overwrite=True,
                        last_grad=gb[1], last_grad_scale=0.5)
        nsg.step_ex(acc, mom, mst, lay.params, lay.parts, 0.95, 0.02, method, 5, 0.05, mode, **opts)
        out[name] = [x.cpu().numpy() for x in (acc, mom, mst)]
    return out


def child(path):
    """Runs in a fresh process with the debug library."""
    import torch
    nsg.use_library(nsg.DEBUG_LIB_PATH)
    res = run_cases(torch)
    errors = [nsg.device_error()]
    lay = wl.tiny_layout()
    acc = torch.zeros(lay.storage_size, dtype=torch.float32, device="cuda")
    g = torch.zeros(lay.storage_size, dtype=torch.bfloat16, device="cuda")
    with nsg.testing(extent_shrink=64):
        nsg.accumulate(acc, g, 1.0, params=lay.params, parts=lay.parts)
        errors.append(nsg.device_error())
    errors.append(nsg.device_error())
    with nsg.testing(extent_shrink=64):
        nsg.accumulate_n(acc, [g, g], 1.0, params=lay.params, parts=lay.parts)
        errors.append(nsg.device_error())
    errors.append(nsg.device_error())
    np.savez(path, errors=np.array(errors), **{f"{k}/{i}": v for k, vs in res.items()
                                                for i, v in enumerate(vs)})


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    nsg.build(debug=True)
    return t


def test_debug_build_reports_nothing_and_matches_release(torch, tmp_path):
    path = str(tmp_path / "debug.npz")
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_gpu_debug_build as t; t.child(%r)" % (HERE, os.path.dirname(HERE), path))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    d = np.load(path)
    errors = d["errors"].tolist()
    assert errors[0] == 0, errors        # every tile of every case in bounds
    assert errors[1] == 16, errors       # the planted short extent is reported
    assert errors[2] == 0, errors        # and cleared once read
    assert errors[3:] == [16, 0], errors  # the same for muon_accumulate_n
    want = run_cases(torch)
    for name, bufs in want.items():
        for i, w in enumerate(bufs):
            assert np.array_equal(bits(d[f"{name}/{i}"]), bits(w)), (name, i)
    assert nsg.device_error() == 0
