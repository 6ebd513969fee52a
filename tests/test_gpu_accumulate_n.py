"""muon_accumulate_n (several bf16 micro-batches accumulated in one pass):
bit for bit the result of muon_accumulate on each micro-batch in order, the
first with `overwrite` -- over the partition tables (16-byte runs and
element-wise ragged ones; padding sentinels untouched) and densely over n
elements (a length that is not a multiple of 4) -- and the oracle's
accumulate chain ("Support Muon in BF16_Optimizer with FP32 gradient
accumulation", PR description: FP32 accumulation of BF16 micro-batches)."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import oracle.bf16 as obf
import oracle.muon as om
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


def layout():
    """Muon blocks of both orientations, odd-sized auxiliary groups and
    shuffled storage over 3 partitions: aligned and ragged runs."""
    return wl.build_layout(
        [[wl.ParamSpec("wq", 128, 192, 4), wl.ParamSpec("wt", 192, 128)],
         [wl.ParamSpec("ln", 1, 769, use_muon=False), wl.ParamSpec("odd", 7, 5, use_muon=False)],
         [wl.ParamSpec("w17", 17, 13)]], 128, 3, "shuffled", 5)


@pytest.mark.parametrize("count", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("overwrite", [False, True])
def test_tables_match_sequential_accumulates(torch, count, overwrite):
    lay = layout()
    grads = micro_batch_grads(lay, 40 + count, 0, count, wl.loguniform_sigmas(lay, 40, 1e-3, 1e-1))
    gb = [bf16_tensor(wl.bf16_storage_grad(lay, g), torch) for g in grads]
    start = wl.storage_with_sentinels(lay, wl.gaussian_grads(lay, 41, 0, None, bf16=False))
    scales = [1.0 / (j + 3) for j in range(count)]
    a0, a1 = to_dev(start, torch), to_dev(start, torch)
    for j in range(count):
        nsg.accumulate(a0, gb[j], scales[j], overwrite=overwrite and j == 0, params=lay.params,
                       parts=lay.parts)
    nsg.accumulate_n(a1, gb, scales, overwrite=overwrite, params=lay.params, parts=lay.parts)
    got, want = a1.cpu().numpy(), a0.cpu().numpy()
    np.testing.assert_array_equal(bits(got), bits(want))
    pad = wl.padding_mask(lay)
    assert (bits(got)[pad] == wl.NAN_SENTINEL_BITS).all()
    # and the oracle's chain on the covered elements
    acc = None if overwrite else np.where(pad, 0, start).astype(np.float32)
    for j in range(count):
        g = obf.bits_to_f32(wl.bf16_storage_grad(lay, grads[j]))
        acc = om.accumulate(acc, g, np.float32(scales[j]), overwrite=(overwrite and j == 0))
    np.testing.assert_array_equal(bits(got[~pad]), bits(acc[~pad]))


@pytest.mark.parametrize("count", [2, 4])
def test_dense_matches_sequential_accumulates(torch, count):
    n = 3 * 32768 + 4099
    rng = np.random.default_rng(77)
    gb = [torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16).cuda()
          for _ in range(count)]
    start = rng.standard_normal(n).astype(np.float32)
    for overwrite in (False, True):
        a0, a1 = to_dev(start, torch), to_dev(start, torch)
        for j in range(count):
            nsg.accumulate(a0, gb[j], 0.25, overwrite=overwrite and j == 0)
        nsg.accumulate_n(a1, gb, 0.25, overwrite=overwrite)
        np.testing.assert_array_equal(bits(a1.cpu().numpy()), bits(a0.cpu().numpy()))
    assert nsg.device_error() == 0
