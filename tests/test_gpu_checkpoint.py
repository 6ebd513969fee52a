"""Checkpoint and resume: the optimizer's whole state is the caller's
buffers (momentum, master, and the auxiliary Adam moments), so five steps in
a row must equal, bit for bit, two steps, a save of that state to host
memory, a restore into fresh device buffers after the library has dropped
its workspaces and plans, and three more steps ("Support Muon in
BF16_Optimizer with FP32 gradient accumulation": checkpoint continuation is
exact; "Fix Muon optimizer under ZeRO CPU offload ...": state rebound after
a load)."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import bf16_tensor, bits, micro_batch_grads, to_dev

pytestmark = pytest.mark.gpu

BETA, LR, CLIP = 0.95, 0.02, 0.05
GAS, STEPS, SAVE_AT = 2, 5, 2
F = lambda x: float(np.float32(x))   # noqa: E731


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def layout():
    return wl.build_layout(
        [[wl.ParamSpec("wq", 128, 192, 4), wl.ParamSpec("wt", 192, 128)],
         [wl.ParamSpec("ln", 1, 768, use_muon=False), wl.ParamSpec("odd", 7, 5, use_muon=False)],
         [wl.ParamSpec("w17", 17, 13)]], 128, 3, "shuffled", 3)


def initial_state(lay):
    z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
    m = [np.float32(0.01) * x for x in wl.gaussian_grads(lay, 31, 1, None, bf16=False)]
    w = wl.gaussian_grads(lay, 31, 2, None, bf16=False)
    return {"accum": wl.storage_with_sentinels(lay, z), "momentum": wl.storage_with_sentinels(lay, m),
            "master": wl.storage_with_sentinels(lay, w), "exp_avg": wl.storage_with_sentinels(lay, z),
            "exp_avg_sq": wl.storage_with_sentinels(lay, z)}


def run_steps(torch, lay, host_state, first, last, method, mode, adam):
    """Restore host_state into fresh device buffers, run steps [first, last)
    and save the state back to host memory."""
    dev = {k: to_dev(v, torch) for k, v in host_state.items()}
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    results = []
    for k in range(first, last):
        grads = micro_batch_grads(lay, 33, k, GAS, wl.loguniform_sigmas(lay, 33, 1e-3, 1e-1))
        for mb, g in enumerate(grads):
            nsg.accumulate(dev["accum"], bf16_tensor(wl.bf16_storage_grad(lay, g), torch), 1.0 / GAS,
                           overwrite=(mb == 0), params=lay.params, parts=lay.parts)
        ad = None
        if adam:
            ad = dict(lr=F(1e-3), beta1=F(0.9), beta2=F(0.999), eps=F(1e-8), step=k + 1,
                      exp_avg=dev["exp_avg"], exp_avg_sq=dev["exp_avg_sq"])
        nsg.step_ex(dev["accum"], dev["momentum"], dev["master"], lay.params, lay.parts, BETA, LR,
                    method, 5, CLIP, mode, adam=ad, result=res)
        results.append(nsg.read_result(res))
    torch.cuda.synchronize()
    assert nsg.device_error() == 0
    return {k: v.cpu().numpy() for k, v in dev.items()}, results


@pytest.mark.parametrize("method,mode,adam", [("standard", "bf16", False), ("gram", "fp32", True),
                                              ("gram", "bf16", True)])
def test_resume_from_saved_state_is_bit_identical(torch, method, mode, adam):
    lay = layout()
    s0 = initial_state(lay)
    straight, r_straight = run_steps(torch, lay, s0, 0, STEPS, method, mode, adam)
    saved, r_first = run_steps(torch, lay, s0, 0, SAVE_AT, method, mode, adam)
    nsg.release_workspace()   # a restarted process rebuilds its plans
    resumed, r_rest = run_steps(torch, lay, saved, SAVE_AT, STEPS, method, mode, adam)
    assert all(r["applied"] == 1 for r in r_straight)
    assert r_first + r_rest == r_straight
    for name in ("accum", "momentum", "master") + (("exp_avg", "exp_avg_sq") if adam else ()):
        np.testing.assert_array_equal(bits(straight[name]), bits(resumed[name]), err_msg=name)
