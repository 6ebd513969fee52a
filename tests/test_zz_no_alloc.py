"""muon_newton_schulz_noalloc: the Newton-Schulz entry point for callers that
cannot allocate device memory (processes whose device memory belongs to
another allocator, runtimes that forbid allocation once they serve).  It
must agree with muon_newton_schulz and with the oracle on repeated calls that
reuse its one fixed scratch array, at the edges of that array's limits and
when host threads call it concurrently on one stream, and must refuse
matrices beyond the limits.

The two entries run different kernels for FP32 operands and for gram's m x m
recurrence (CUDA-core GEMM here, split-3 tensor-core products there), so they
are compared by the operand mode's tolerance, not bit for bit.

Collected last (file name) so a failure here never hides another test."""

import threading

import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import ORACLE_MODE, assert_close_update, to_dev
from oracle import newton_schulz as ons

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def noalloc(torch, X, method, mode, steps=5, stream=None, Y=None):
    """Calls the C entry point directly (argument marshalling only)."""
    if Y is None:
        Y = torch.empty_like(X)
    io = 0 if X.dtype == torch.bfloat16 else 1
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = nsg.lib().muon_newton_schulz_noalloc(
        X.data_ptr(), Y.data_ptr(), X.shape[0], X.shape[1], io, nsg.NS_METHODS[method], steps,
        nsg.OPERAND_MODES[mode], s.cuda_stream)
    assert rc == 0, nsg.last_error()
    return Y


def make_input(torch, shape, mode, seed):
    """(host values the oracle reads, the device tensor the library reads)."""
    G = wl.rng_for(seed, *shape).standard_normal(shape).astype(np.float32)
    if mode == "bf16":
        G = wl.to_bf16_values(G)
        return G, to_dev(G, torch, torch.bfloat16)
    return G, to_dev(G, torch)


def oracle(G, method, mode, steps=5):
    return ons.newton_schulz(G, method, steps, ORACLE_MODE[mode])


# two calls in a row with different shapes and methods: the second reuses the
# scratch the first left behind
SEQUENCES = [
    [((300, 77), "standard"), ((512, 1000), "gram")],
    [((512, 2048), "gram"), ((64, 768), "standard")],
]


@pytest.mark.parametrize("mode", ["bf16", "fp32"])
@pytest.mark.parametrize("seq", range(len(SEQUENCES)))
def test_noalloc_matches_allocating_entry_and_oracle(torch, mode, seq):
    for k, (shape, method) in enumerate(SEQUENCES[seq]):
        G, X = make_input(torch, shape, mode, 60 + 10 * seq + k)
        got = noalloc(torch, X, method, mode).float().cpu().numpy()
        want = nsg.newton_schulz(X, ns_method=method, operand_mode=mode).float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_close_update(got, want, mode, f"{shape} {method} {mode} call {k} vs allocating")
        assert_close_update(got, oracle(G, method, mode), mode,
                            f"{shape} {method} {mode} call {k} vs oracle")
    assert nsg.device_error() == 0


# the limits exactly: rows*cols = 2^20 with min(rows, cols) = 512, and
# max(rows, cols) = 16384 with m = 64 (tall, so transposed)
EDGE_SHAPES = [(512, 2048), (16384, 64)]


@pytest.mark.parametrize("shape", EDGE_SHAPES)
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_noalloc_at_the_limits(torch, shape, method, mode):
    G, X = make_input(torch, shape, mode, 90)
    got = noalloc(torch, X, method, mode).float().cpu().numpy()
    assert_close_update(got, oracle(G, method, mode), mode, f"{shape} {method} {mode} vs oracle")
    want = nsg.newton_schulz(X, ns_method=method, operand_mode=mode).float().cpu().numpy()
    assert_close_update(got, want, mode, f"{shape} {method} {mode} vs allocating")
    assert nsg.device_error() == 0


def test_noalloc_two_host_threads_one_stream(torch):
    """Two host threads issue interleaved calls of different shapes and
    methods on one shared stream, so the GPU work stays ordered and the
    shared array is never used by two calls at once; the host-side plan
    tables are guarded by the library lock.  Every result matches the
    oracle."""
    stream = torch.cuda.Stream()
    jobs = [[((256, 700), "standard", "bf16"), ((96, 1000), "gram", "bf16"),
             ((400, 300), "gram", "fp32")],
            [((128, 2048), "gram", "bf16"), ((700, 256), "standard", "fp32"),
             ((64, 64), "standard", "bf16")]]
    inputs = [[make_input(torch, shape, mode, 100 + 10 * t + i)
               for i, (shape, _, mode) in enumerate(js)] for t, js in enumerate(jobs)]
    outs = [[torch.empty_like(X) for _, X in ins] for ins in inputs]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(2)

    def worker(t):
        try:
            start.wait()
            for rep in range(3):
                for i, (shape, method, mode) in enumerate(jobs[t]):
                    noalloc(torch, inputs[t][i][1], method, mode, stream=stream, Y=outs[t][i])
        except Exception as e:   # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    stream.synchronize()
    for t in range(2):
        for i, (shape, method, mode) in enumerate(jobs[t]):
            got = outs[t][i].float().cpu().numpy()
            assert_close_update(got, oracle(inputs[t][i][0], method, mode), mode,
                                f"thread {t} {shape} {method} {mode}")
    assert nsg.device_error() == 0


def test_noalloc_repeated_call_same_input_is_stable(torch):
    _, X = make_input(torch, (256, 4096), "bf16", 77)
    a = noalloc(torch, X, "standard", "bf16").float().cpu().numpy()
    b = noalloc(torch, X, "standard", "bf16").float().cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [(1024, 1025), (513, 600), (32, 16385)],
                         ids=["elements", "min dim", "max dim"])
def test_noalloc_rejects_oversized(torch, shape):
    X = torch.zeros(shape, dtype=torch.float32, device="cuda")
    Y = torch.empty_like(X)
    rc = nsg.lib().muon_newton_schulz_noalloc(X.data_ptr(), Y.data_ptr(), shape[0], shape[1], 1, 0,
                                              5, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == nsg.MUON_ERR_UNSUPPORTED
    assert "too large" in nsg.last_error()
