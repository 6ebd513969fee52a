"""A whole optimizer step -- the micro-batch accumulations and muon_step_ex
(with the folded last micro-batch; or all micro-batches in one
muon_accumulate_n pass and the plain step; or two micro-batches folded
with overwrite, the gradient formed by every pass) -- recorded into a CUDA graph once its
plans exist, then replayed: the library issues only stream-ordered work on
the caller's stream in steady state (no allocation, no synchronisation,
no host reads), so the replays must leave accum, momentum, master and the
result bit-identical to the same steps run eagerly."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import bf16_tensor, bits, micro_batch_grads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


@pytest.mark.parametrize("method,mode,flow", [("standard", "bf16", "fold_last"),
                                              ("gram", "fp32", "fold_last"),
                                              ("standard", "bf16", "accumulate_n"),
                                              ("gram", "bf16", "fold_both")])
def test_step_replays_from_a_cuda_graph(torch, method, mode, flow):
    lay = wl.build_layout([[wl.ParamSpec("q", 256, 256, 4), wl.ParamSpec("up", 512, 256),
                            wl.ParamSpec("down", 256, 512)],
                           [wl.ParamSpec("ln", 1, 256, use_muon=False)]], 128, 4)
    gas = 2 if flow == "fold_both" else 3
    grads = micro_batch_grads(lay, 21, 0, gas, wl.loguniform_sigmas(lay, 21, 1e-3, 1e-1))
    gb = [bf16_tensor(wl.bf16_storage_grad(lay, g), torch) for g in grads]
    m0 = wl.storage_with_sentinels(lay, [np.float32(0.01) * x for x in
                                         wl.gaussian_grads(lay, 22, 1, None, bf16=False)])
    w0 = wl.storage_with_sentinels(lay, wl.gaussian_grads(lay, 22, 2, None, bf16=False))
    a0 = wl.storage_with_sentinels(lay, [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs])

    def fresh():
        return to_dev(a0, torch), to_dev(m0, torch), to_dev(w0, torch), \
            torch.zeros(4, dtype=torch.int32, device="cuda")

    def one_step(acc, mom, mst, res, stream):
        if flow == "fold_last":
            for mb in range(gas - 1):
                nsg.accumulate(acc, gb[mb], 1.0 / gas, overwrite=(mb == 0), params=lay.params,
                               parts=lay.parts, stream=stream)
            opts = dict(last_grad=gb[-1], last_grad_scale=1.0 / gas)
        elif flow == "accumulate_n":
            nsg.accumulate_n(acc, gb, 1.0 / gas, overwrite=True, params=lay.params,
                             parts=lay.parts, stream=stream)
            opts = {}
        else:
            opts = dict(prev_grad=gb[0], prev_grad_scale=0.5, prev_grad_overwrite=True,
                        last_grad=gb[1], last_grad_scale=0.5)
        nsg.step_ex(acc, mom, mst, lay.params, lay.parts, 0.95, 0.02, method, 5, 0.05, mode,
                    result=res, stream=stream, **opts)

    # eager: two steps (the first also builds the plans)
    e = fresh()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):
            one_step(*e, s)
    torch.cuda.synchronize()
    # graph: the same two steps as two replays of one recorded step
    g = fresh()
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=cs):
        one_step(*g, cs)
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert nsg.device_error() == 0
    assert nsg.read_result(e[3]) == nsg.read_result(g[3])
    assert nsg.read_result(g[3])["applied"] == 1
    for x, y in zip(e[:3], g[:3]):
        np.testing.assert_array_equal(bits(x.cpu().numpy()), bits(y.cpu().numpy()))
