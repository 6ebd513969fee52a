"""The data-parallel step's kernels on the GPU: several ranks' phases run in
one process on one GPU, one rank after another, with the buffers of the two
all-to-all exchanges and the all-reduce moved between the ranks by the test
(no kernel waits on another rank's).  Every rank holds only its own
partitions; the result is compared with the single-GPU step on the whole
flat buffer (the partition table emulating the same ranks) and with the
oracle:

* momentum bit for bit (m' = beta m + g is the same FP32 arithmetic at the
  owner);
* the update of every parameter by the operand mode's rule against the
  oracle (BF16: rel-F <= 1e-2 against the BF16-emulating oracle; FP32: atol
  1e-4 / rtol 1e-3 against the exact oracle), after dividing out the clip
  coefficient;
* the global norm and the clip coefficient within 1e-5 of the single-GPU
  step's (the sums of squares are added in another order);
* the master weights within the write-back's rounding of the single-GPU
  step's; padding bit for bit untouched; a non-finite gradient on any rank
  skips the step on every rank."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
from newton_schulz_fp32_gb300 import dp
import workloads as wl
from harness import ORACLE_MODE, assert_close_update, bits
from oracle import muon as om

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def part_ranks(lay):
    return np.arange(len(lay.parts), dtype=np.int32) % lay.nparts


def local_view(lay, parts_local, pr, rank, glob, size):
    out = np.zeros(size, np.float32)
    for p in range(len(lay.parts)):
        if pr[p] == rank:
            n = int(lay.parts["flat_end"][p] - lay.parts["flat_begin"][p])
            g0, l0 = int(lay.parts["storage_offset"][p]), int(parts_local["storage_offset"][p])
            out[l0:l0 + n] = glob[g0:g0 + n]
    return out


def emulated_dp_step(torch, lay, world, acc, mom, mst, method, mode, clip=CLIP, assign="balanced",
                     grad_scale=1.0, budget=0):
    """Runs the data-parallel step of `world` ranks in this process; acc,
    mom, mst are whole-model storage buffers (numpy); returns each rank's
    buffers after the step and each rank's result."""
    pr = part_ranks(lay)
    parts_local, sizes = dp.local_partition_table(lay.parts, pr, world)
    ranks = []
    for r in range(world):
        plan = dp.DPPlan(lay.params, parts_local, pr, world, r, method, assign)
        bufs = [torch.from_numpy(local_view(lay, parts_local, pr, r, g, sizes[r])).cuda()
                for g in (acc, mom, mst)]
        ranks.append((plan, dp.DataParallelMuon(plan, workspace_budget=budget), bufs,
                      torch.zeros(4, dtype=torch.int32, device="cuda")))
    off = lambda counts: np.concatenate([[0], np.cumsum(counts)])
    # 1. pack, all-to-all
    for plan, d, (a, m, w), res in ranks:
        d.pack_forward(a, m)
    torch.cuda.synchronize()
    for s, (ps, ds, _, _) in enumerate(ranks):
        so = off(ps.send_counts)
        for t, (pt, dt, _, _) in enumerate(ranks):
            ro = off(pt.recv_counts)
            n = int(ps.send_counts[t])
            dt.recv[ro[s]:ro[s] + n].copy_(ds.send[so[t]:so[t] + n])
    # 2. owners' step, all-reduce of the statistics
    for plan, d, _, _ in ranks:
        d.local_step(BETA, method, 5, mode, grad_scale)
    torch.cuda.synchronize()
    total = sum(d.stats.clone() for _, d, _, _ in ranks)
    for _, d, _, _ in ranks:
        d.stats.copy_(total)
    # 3. pack back, reverse all-to-all (split sizes swapped)
    for _, d, _, _ in ranks:
        d.pack_reverse()
    torch.cuda.synchronize()
    for t, (pt, dt, _, _) in enumerate(ranks):
        so = off(pt.recv_counts)
        for s, (ps, ds, _, _) in enumerate(ranks):
            ro = off(ps.send_counts)
            n = int(pt.recv_counts[s])
            ds.send[ro[t]:ro[t] + n].copy_(dt.recv[so[s]:so[s] + n])
    # 4. write-back
    for plan, d, (a, m, w), res in ranks:
        d.finish(a, m, w, LR, clip, res)
    torch.cuda.synchronize()
    out = [[b.cpu().numpy() for b in bufs] + [nsg.read_result(res)] for _, _, bufs, res in ranks]
    for plan, _, _, _ in ranks:
        plan.close()
    return out, parts_local, sizes, pr


def whole_step(torch, lay, acc, mom, mst, method, mode, clip=CLIP, grad_scale=1.0):
    bufs = [torch.from_numpy(x.copy()).cuda() for x in (acc, mom, mst)]
    res = nsg.read_result(nsg.step_ex(*bufs, lay.params, lay.parts, BETA, LR, method, 5, clip, mode,
                                      grad_scale=grad_scale))
    return [b.cpu().numpy() for b in bufs] + [res]


def make_state(lay, seed, nan=False):
    grads = wl.gaussian_grads(lay, seed, 0, wl.loguniform_sigmas(lay, seed, 1e-3, 1e-1))
    if nan:
        grads[-1][0, 0] = np.inf
    m0 = [0.1 * g for g in wl.gaussian_grads(lay, seed, 1, None, bf16=False)]
    w0 = wl.gaussian_grads(lay, seed, 2, None, bf16=False)
    return (wl.storage_with_sentinels(lay, grads), wl.storage_with_sentinels(lay, m0),
            wl.storage_with_sentinels(lay, w0))


CASES = [("tiny", 2, "gram", "bf16", {}), ("tiny", 3, "standard", "fp32", {}),
         ("gpt2_layer", 2, "standard", "bf16", {}), ("gpt2_layer", 4, "gram", "fp32", {}),
         ("gpt2_layer", 3, "gram", "bf16", {}),
         # a loss scale undone (2^-3) and the owners' NS in waves of one block
         ("gpt2_layer", 3, "standard", "bf16", {"grad_scale": 0.125, "budget": 1}),
         ("tiny", 2, "gram", "fp32", {"grad_scale": 0.5, "budget": 1})]
LAYOUTS = {"tiny": lambda w: wl.tiny_layout(nparts=w),
           "gpt2_layer": lambda w: wl.gpt2_small_layout(layers=1, nparts=w)}


@pytest.mark.parametrize("name,world,method,mode,opts", CASES)
def test_emulated_ranks_match_whole_step_and_oracle(torch, name, world, method, mode, opts):
    lay = LAYOUTS[name](world)
    acc, mom, mst = make_state(lay, 900 + world)
    gs = opts.get("grad_scale", 1.0)
    ranks, parts_local, sizes, pr = emulated_dp_step(torch, lay, world, acc, mom, mst, method, mode,
                                                     grad_scale=gs, budget=opts.get("budget", 0))
    ref = whole_step(torch, lay, acc, mom, mst, method, mode, grad_scale=gs)
    ores = om.muon_step_flat(acc, mom, mst, lay.params, lay.parts, BETA, LR, method, 5, CLIP,
                             ORACLE_MODE[mode], grad_scale=gs)
    r0 = ranks[0][3]
    assert all(r[3]["applied"] == 1 for r in ranks)
    assert all(r[3] == r0 for r in ranks)          # every rank reports the same step
    assert r0["ns_calls"] == ref[3]["ns_calls"]
    assert abs(r0["global_norm"] - ref[3]["global_norm"]) <= 1e-5 * ref[3]["global_norm"]
    assert abs(r0["clip_coef"] - ref[3]["clip_coef"]) <= 1e-5 * ref[3]["clip_coef"]
    mask = wl.padding_mask(lay)
    for r in range(world):
        a, m, w, _ = ranks[r]
        want = [local_view(lay, parts_local, pr, r, x, sizes[r]) for x in ref[:3]]
        pad = local_view(lay, parts_local, pr, r, mask.astype(np.float32), sizes[r]) > 0
        assert np.array_equal(bits(m), bits(want[1]))                       # momentum
        for got, w_ in ((a, want[0]), (m, want[1]), (w, want[2])):          # padding untouched
            assert np.array_equal(bits(got)[pad], bits(w_)[pad])
        # master: the same write-back of updates that agree within the mode's rule
        scale = np.abs(want[2][~pad]) + LR * np.abs(want[0][~pad]) + 1e-30
        tol = 1e-6 if mode == "fp32" else 2e-2
        assert np.all(np.abs(w[~pad] - want[2][~pad]) <= tol * scale + 1e-7)
    # updates of every parameter against the oracle (clip coefficient divided out)
    full = np.zeros_like(acc)
    for r in range(world):
        for p in range(len(lay.parts)):
            if pr[p] == r:
                n = int(lay.parts["flat_end"][p] - lay.parts["flat_begin"][p])
                g0, l0 = int(lay.parts["storage_offset"][p]), int(parts_local["storage_offset"][p])
                full[g0:g0 + n] = ranks[r][0][l0:l0 + n]
    got = wl.unpack(lay, full)
    want = wl.unpack(lay, ores[0])
    for k, spec in enumerate(lay.specs):
        if spec.use_muon:
            assert_close_update(got[k] / r0["clip_coef"], want[k] / ores[3]["coef"], mode,
                                f"{name} {spec.name}")
    assert nsg.device_error() == 0


def test_emulated_ranks_skip_together_on_overflow(torch):
    lay = wl.gpt2_small_layout(layers=1, nparts=3)
    acc, mom, mst = make_state(lay, 950, nan=True)
    ranks, parts_local, sizes, pr = emulated_dp_step(torch, lay, 3, acc, mom, mst, "standard", "bf16")
    for r in range(3):
        assert ranks[r][3]["applied"] == 0
        for got, x in zip(ranks[r][:3], (acc, mom, mst)):
            assert np.array_equal(bits(got), bits(local_view(lay, parts_local, pr, r, x, sizes[r])))
