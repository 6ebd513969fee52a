"""muon_newton_schulz_noalloc: the Newton-Schulz entry point for callers that
cannot allocate device memory (stream capture, foreign allocators, runtimes
that forbid allocation after start-up).  It must give the same results as
muon_newton_schulz, on repeated calls that reuse its one fixed scratch
array, and must refuse matrices beyond that array's limits.

Collected last (file name) so a failure here never hides another test."""

import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import assert_close_update, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def noalloc(torch, X, method, mode, steps=5):
    """Calls the C entry point directly (argument marshalling only)."""
    Y = torch.empty_like(X)
    io = 0 if X.dtype == torch.bfloat16 else 1
    rc = nsg.lib().muon_newton_schulz_noalloc(
        X.data_ptr(), Y.data_ptr(), X.shape[0], X.shape[1], io, nsg.NS_METHODS[method], steps,
        nsg.OPERAND_MODES[mode], torch.cuda.current_stream().cuda_stream)
    assert rc == 0, nsg.last_error()
    return Y


def make_input(torch, shape, mode, seed):
    G = wl.rng_for(seed, *shape).standard_normal(shape).astype(np.float32)
    if mode == "bf16":
        return to_dev(wl.to_bf16_values(G), torch, torch.bfloat16)
    return to_dev(G, torch)


# two calls in a row with different shapes and methods: the second reuses the
# scratch the first left behind
SEQUENCES = [
    [((300, 77), "standard"), ((512, 1000), "gram")],
    [((512, 2048), "gram"), ((64, 768), "standard")],
]


@pytest.mark.parametrize("mode", ["bf16", "fp32"])
@pytest.mark.parametrize("seq", range(len(SEQUENCES)))
def test_noalloc_matches_allocating_entry(torch, mode, seq):
    for k, (shape, method) in enumerate(SEQUENCES[seq]):
        X = make_input(torch, shape, mode, 60 + 10 * seq + k)
        got = noalloc(torch, X, method, mode).float().cpu().numpy()
        want = nsg.newton_schulz(X, ns_method=method, operand_mode=mode).float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_close_update(got, want, mode, f"{shape} {method} {mode} call {k}")
    assert nsg.device_error() == 0


def test_noalloc_repeated_call_same_input_is_stable(torch):
    X = make_input(torch, (256, 4096), "bf16", 77)
    a = noalloc(torch, X, "standard", "bf16").float().cpu().numpy()
    b = noalloc(torch, X, "standard", "bf16").float().cpu().numpy()
    assert np.array_equal(a, b)


def test_noalloc_rejects_oversized(torch):
    X = torch.zeros((1024, 1025), dtype=torch.float32, device="cuda")
    Y = torch.empty_like(X)
    rc = nsg.lib().muon_newton_schulz_noalloc(X.data_ptr(), Y.data_ptr(), 1024, 1025, 1, 0, 5, 1,
                                              torch.cuda.current_stream().cuda_stream)
    assert rc == nsg.MUON_ERR_UNSUPPORTED
    assert "too large" in nsg.last_error()
