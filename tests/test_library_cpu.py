"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol the header declares, and rejects bad tables and arguments on
the host before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20   # a non-NULL, aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    nsg.build()
    return nsg.lib()


def header_symbols():
    with open(os.path.join(ROOT, "include", "muon.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"MUON_API\s+[\w\s\*]+?\b(muon_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 9
    assert sorted(nsg.EXPORTED) == syms
    for s in syms:
        assert hasattr(lib, s), s


def test_struct_sizes_match_header():
    assert nsg.PARAM_DTYPE.itemsize == 24 and nsg.PART_DTYPE.itemsize == 24
    assert nsg.PARAM_DTYPE == wl.PARAM_DTYPE and nsg.PART_DTYPE == wl.PART_DTYPE
    assert ctypes.sizeof(nsg.Stats) == 48 and ctypes.sizeof(nsg.PhaseTime) == 32


def _step(lib, params, parts, **kw):
    args = dict(beta=0.95, lr=0.02, method=0, steps=5, clip=0.0, mode=0)
    args.update(kw)
    p = np.ascontiguousarray(params, dtype=nsg.PARAM_DTYPE)
    q = np.ascontiguousarray(parts, dtype=nsg.PART_DTYPE)
    return lib.muon_step(FAKE, FAKE, FAKE, p.ctypes.data if len(p) else None, len(p),
                         q.ctypes.data if len(q) else None, len(q), args["beta"], args["lr"],
                         args["method"], args["steps"], args["clip"], args["mode"], FAKE, None)


def test_invalid_tables_rejected_on_host(lib):
    lay = wl.tiny_layout()
    P, Q = lay.params.copy(), lay.parts.copy()
    cases = []
    bad = P.copy(); bad["offset"][1] = 100                       # overlaps the first matrix
    cases.append((bad, Q, "overlap"))
    bad = P.copy(); bad["offset"][0] = lay.flat_size - 5         # runs past the partitions
    cases.append((bad, Q, "covered"))
    bad = P.copy(); bad["rows"][0] = 0
    cases.append((bad, Q, "rows or cols"))
    bad = P.copy(); bad["num_heads"][0] = 4                      # 17 % 4 != 0
    cases.append((bad, Q, "num_heads"))
    badq = Q.copy(); badq[[0, 1]] = badq[[1, 0]]                 # unsorted
    cases.append((P, badq, "sorted"))
    badq = Q.copy(); badq["storage_offset"][1] = 50              # storage overlap
    cases.append((P, badq, "storage"))
    badq = Q.copy(); badq["flat_end"][0] = 100                   # hole inside the first matrix
    cases.append((P, badq, "covered"))
    for params, parts, word in cases:
        rc = _step(lib, params, parts)
        assert rc == nsg.MUON_ERR_INVALID, (word, rc)
        assert word in lib.muon_last_error().decode(), lib.muon_last_error()


def test_unsupported_arguments(lib):
    lay = wl.tiny_layout()
    assert _step(lib, lay.params, lay.parts, steps=0) == nsg.MUON_ERR_UNSUPPORTED
    assert _step(lib, lay.params, lay.parts, method=7) == nsg.MUON_ERR_UNSUPPORTED
    assert _step(lib, lay.params, lay.parts, mode=3) == nsg.MUON_ERR_UNSUPPORTED
    assert _step(lib, lay.params, lay.parts, lr=float("nan")) == nsg.MUON_ERR_INVALID


def test_valid_tables_without_gpu_fail_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lay = wl.gpt2_small_layout(layers=1)
    assert _step(lib, lay.params, lay.parts) == nsg.MUON_ERR_CUDA
    assert lib.muon_last_error().decode() != ""


def test_python_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(nsg, "_lib", None)
    monkeypatch.setattr(nsg, "LIB_PATH", "/nonexistent/libmuon.so")
    with pytest.raises(nsg.MuonError):
        nsg.lib()


def _step_ex(lib, opts, ptrs=(FAKE, FAKE, FAKE)):
    lay = wl.tiny_layout()
    p = np.ascontiguousarray(lay.params, dtype=nsg.PARAM_DTYPE)
    q = np.ascontiguousarray(lay.parts, dtype=nsg.PART_DTYPE)
    return lib.muon_step_ex(*ptrs, p.ctypes.data, len(p), q.ctypes.data, len(q), 0.95, 0.02, 1, 5,
                            0.0, 0, ctypes.byref(opts) if opts is not None else None, FAKE, None)


def test_step_options_struct_layout():
    # muon.h: the original layout ends at workspace_budget (64 bytes); the
    # folded last micro-batch follows it (80), then the statistics pointer
    assert ctypes.sizeof(nsg.StepOptions) == 104
    assert nsg.StepOptions.adam_step.offset == 32 and nsg.StepOptions.workspace_budget.offset == 56
    assert nsg.StepOptions.last_grad.offset == nsg.STEP_OPTIONS_V1_SIZE == 64
    assert nsg.StepOptions.last_grad_scale.offset == 72
    assert nsg.StepOptions.last_grad_overwrite.offset == 76
    assert nsg.StepOptions.stats_out.offset == nsg.STEP_OPTIONS_V2_SIZE == 80
    assert nsg.StepOptions.prev_grad.offset == 88
    assert nsg.StepOptions.prev_grad_scale.offset == 96
    assert nsg.StepOptions.prev_grad_overwrite.offset == 100


def test_step_options_rejected_on_host(lib):
    adam = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=1, exp_avg=FAKE, exp_avg_sq=FAKE)
    cases = []
    o = nsg.step_options(); o.struct_size = 8
    cases.append((o, "struct_size"))
    cases.append((nsg.step_options(clip_mode=5), "clip_mode"))
    cases.append((nsg.step_options(grad_scale=-1.0), "grad_scale"))
    cases.append((nsg.step_options(grad_scale=float("inf")), "grad_scale"))
    cases.append((nsg.step_options(adam=dict(adam, exp_avg=None)), "exp_avg"))
    cases.append((nsg.step_options(adam=dict(adam, exp_avg_sq=FAKE + 4)), "aligned"))
    cases.append((nsg.step_options(adam=dict(adam, step=0)), "adam_step"))
    cases.append((nsg.step_options(adam=dict(adam, beta2=1.0)), "betas"))
    cases.append((nsg.step_options(adam=dict(adam, eps=-1.0)), "adam_eps"))
    cases.append((nsg.step_options(last_grad=FAKE + 2), "8-byte"))
    cases.append((nsg.step_options(last_grad=FAKE, last_grad_scale=float("nan")), "last_grad_scale"))
    o = nsg.step_options(last_grad=FAKE); o.last_grad_overwrite = 2
    cases.append((o, "last_grad_overwrite"))
    o = nsg.step_options(); o.struct_size = 72
    cases.append((o, "struct_size"))
    cases.append((nsg.step_options(stats_out=FAKE + 4), "stats_out"))
    cases.append((nsg.step_options(prev_grad=FAKE), "needs last_grad"))
    cases.append((nsg.step_options(last_grad=FAKE, prev_grad=FAKE + 2), "8-byte"))
    cases.append((nsg.step_options(last_grad=FAKE, prev_grad=FAKE, prev_grad_scale=float("inf")),
                  "prev_grad_scale"))
    o = nsg.step_options(last_grad=FAKE, prev_grad=FAKE); o.prev_grad_overwrite = 3
    cases.append((o, "prev_grad_overwrite"))
    for opts, word in cases:
        rc = _step_ex(lib, opts)
        assert rc == nsg.MUON_ERR_INVALID, (word, rc)
        assert word in lib.muon_last_error().decode(), lib.muon_last_error()


def test_step_buffers_must_be_16_byte_aligned(lib):
    for ptrs in ((FAKE + 4, FAKE, FAKE), (FAKE, FAKE + 8, FAKE), (FAKE, FAKE, FAKE + 12)):
        assert _step_ex(lib, None, ptrs) == nsg.MUON_ERR_INVALID
        assert "16-byte" in lib.muon_last_error().decode()


def test_valid_options_without_gpu_fail_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    adam = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=3, exp_avg=FAKE, exp_avg_sq=FAKE)
    v1 = nsg.step_options(last_grad=FAKE + 2)   # ignored: the fields are absent in a v1 struct
    v1.struct_size = nsg.STEP_OPTIONS_V1_SIZE
    v2 = nsg.step_options(stats_out=FAKE + 4)   # ignored: absent in a v2 struct
    v2.struct_size = nsg.STEP_OPTIONS_V2_SIZE
    for opts in (None, nsg.step_options(), nsg.step_options("grad", 2.0 ** -10, adam),
                 nsg.step_options(last_grad=FAKE, last_grad_scale=0.25), v1, v2,
                 nsg.step_options(stats_out=FAKE)):
        assert _step_ex(lib, opts) == nsg.MUON_ERR_CUDA


def test_accumulate_n_arguments_rejected_on_host(lib):
    """muon_accumulate_n checks its micro-batch list before any CUDA call."""
    def call(ptrs, count, accum=FAKE):
        grads = (ctypes.c_void_p * max(len(ptrs), 1))(*ptrs)
        scales = (ctypes.c_float * max(len(ptrs), 1))(*([0.5] * len(ptrs)))
        return lib.muon_accumulate_n(accum, ctypes.cast(grads, ctypes.c_void_p),
                                     ctypes.cast(scales, ctypes.c_void_p), count, 1024, 1,
                                     None, 0, None, 0, None)
    assert nsg.ACCUMULATE_MAX == 8
    for ptrs, count, word in [([FAKE], 0, "count"), ([FAKE] * 9, 9, "count"),
                              ([FAKE, None], 2, "grads"), ([FAKE, FAKE + 4], 2, "grads")]:
        assert call(ptrs, count) == nsg.MUON_ERR_INVALID, word
        assert word in lib.muon_last_error().decode(), lib.muon_last_error()
    assert call([FAKE], 1, accum=FAKE + 8) == nsg.MUON_ERR_INVALID
    assert "aligned" in lib.muon_last_error().decode()
    with pytest.raises(ValueError):
        nsg.accumulate_n(FAKE, [FAKE, FAKE], [0.5], n=16)
