"""Python binding of libmuon, the Muon optimizer step on one GB300 GPU.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libmuon.so`` (built in-tree by :func:`build`).  PyTorch tensors
are accepted for device buffers and the current CUDA stream; plain integer
device addresses work too.  There is no CPU fallback: if the library is
missing or the call fails, a :class:`MuonError` is raised.

Table formats match the C structs of ``include/muon.h``:
``PARAM_DTYPE`` ``{int64 offset; int32 rows, cols, num_heads, use_muon}`` and
``PART_DTYPE`` ``{int64 flat_begin, flat_end, storage_offset}``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmuon.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libmuon_debug.so")

PARAM_DTYPE = np.dtype([("offset", "<i8"), ("rows", "<i4"), ("cols", "<i4"),
                        ("num_heads", "<i4"), ("use_muon", "<i4")])
PART_DTYPE = np.dtype([("flat_begin", "<i8"), ("flat_end", "<i8"),
                       ("storage_offset", "<i8")])

MUON_OK, MUON_ERR_INVALID, MUON_ERR_UNSUPPORTED, MUON_ERR_CUDA, MUON_ERR_OOM = 0, -1, -2, -3, -4
NS_METHODS = {"standard": 0, "gram": 1}
OPERAND_MODES = {"bf16": 0, "fp32": 1}
DTYPES = {"bf16": 0, "fp32": 1}
PHASES = ["accumulate", "reduce", "gather", "ns_gemm", "norm", "scatter"]

# Every symbol include/muon.h declares.
EXPORTED = ["muon_accumulate", "muon_accumulate_n", "muon_step", "muon_newton_schulz", "muon_get_stats",
            "muon_last_error", "muon_release_workspace", "muon_device_error",
            "muon_profile_enable", "muon_profile_read", "muon_newton_schulz_noalloc",
            "muon_step_ex", "muon_profile_enable_phases", "muon_describe_tables",
            "muon_testing_set", "muon_dp_plan_create", "muon_dp_plan_destroy",
            "muon_dp_plan_sizes", "muon_dp_plan_tables", "muon_dp_pack", "muon_dp_unpack",
            "muon_dp_finish"]
CLIP_MODES = {"update": 0, "grad": 1}


class MuonError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmuon error {code}: {msg}")
        self.code = code


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("ns_calls_last_step", ctypes.c_int64),
                ("muon_matrices", ctypes.c_int64), ("kernel_launches_last_call", ctypes.c_int64),
                ("kernel_launches_total", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t)]


class StepOptions(ctypes.Structure):
    """muon_step_options_t."""
    _fields_ = [("struct_size", ctypes.c_int32), ("clip_mode", ctypes.c_int32),
                ("grad_scale", ctypes.c_float), ("aux_adam", ctypes.c_int32),
                ("adam_lr", ctypes.c_float), ("adam_beta1", ctypes.c_float),
                ("adam_beta2", ctypes.c_float), ("adam_eps", ctypes.c_float),
                ("adam_step", ctypes.c_int64), ("exp_avg", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("workspace_budget", ctypes.c_uint64),
                ("last_grad", ctypes.c_void_p), ("last_grad_scale", ctypes.c_float),
                ("last_grad_overwrite", ctypes.c_int32), ("stats_out", ctypes.c_void_p),
                ("prev_grad", ctypes.c_void_p), ("prev_grad_scale", ctypes.c_float),
                ("prev_grad_overwrite", ctypes.c_int32)]


STEP_OPTIONS_V1_SIZE = 64   # struct_size of the layout that ends at workspace_budget
STEP_OPTIONS_V2_SIZE = 80   # struct_size of the layout that ends at last_grad_overwrite


class TableInfo(ctypes.Structure):
    """muon_table_info_t."""
    _fields_ = [("muon_params", ctypes.c_int64), ("muon_blocks", ctypes.c_int64),
                ("ns_problems", ctypes.c_int64), ("pair_engine", ctypes.c_int32),
                ("stack_rows", ctypes.c_int32), ("muon_elements", ctypes.c_int64),
                ("aux_elements", ctypes.c_int64), ("padding_elements", ctypes.c_int64),
                ("segments", ctypes.c_int64), ("workspace_bytes", ctypes.c_uint64)]


class PhaseTime(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("total_ms", ctypes.c_double),
                ("algorithmic_bytes", ctypes.c_double), ("algorithmic_flops", ctypes.c_double)]


_lib = None


def build(force: bool = False, verbose: bool = False, debug: bool = False):
    from . import builder as _b
    return _b.build(force=force, verbose=verbose, debug=debug)


def use_library(path: str):
    """Load `path` (e.g. DEBUG_LIB_PATH, the bounds-checking build) instead
    of libmuon.so; only before the library's first use in this process."""
    global LIB_PATH
    if _lib is not None:
        raise MuonError(MUON_ERR_INVALID, "the library is already loaded in this process")
    LIB_PATH = path


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MuonError(MUON_ERR_UNSUPPORTED,
                            f"{LIB_PATH} is missing; build it with newton_schulz_fp32_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.muon_accumulate.argtypes = [P, P, I64, F, I, P, I, P, I, P]
        L.muon_accumulate_n.argtypes = [P, P, P, I, I64, I, P, I, P, I, P]
        L.muon_step.argtypes = [P, P, P, P, I, P, I, F, F, I, I, F, I, P, P]
        L.muon_step_ex.argtypes = [P, P, P, P, I, P, I, F, F, I, I, F, I,
                                   ctypes.POINTER(StepOptions), P, P]
        L.muon_newton_schulz.argtypes = [P, P, I, I, I, I, I, I, P]
        L.muon_newton_schulz_noalloc.argtypes = [P, P, I, I, I, I, I, I, P]
        L.muon_get_stats.argtypes = [ctypes.POINTER(Stats)]
        L.muon_last_error.restype = ctypes.c_char_p
        L.muon_release_workspace.restype = None
        L.muon_profile_enable.argtypes = [I]
        L.muon_profile_enable_phases.argtypes = [ctypes.c_uint32]
        L.muon_describe_tables.argtypes = [P, I, P, I, I, I, ctypes.POINTER(TableInfo)]
        L.muon_profile_read.argtypes = [ctypes.POINTER(PhaseTime), I, I]
        L.muon_testing_set.argtypes = [I, I]
        for name in ("muon_accumulate", "muon_accumulate_n", "muon_step", "muon_step_ex",
                     "muon_newton_schulz", "muon_newton_schulz_noalloc", "muon_get_stats",
                     "muon_device_error", "muon_profile_enable", "muon_profile_read",
                     "muon_profile_enable_phases", "muon_describe_tables",
                     "muon_testing_set"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(rc: int):
    if rc != MUON_OK:
        raise MuonError(rc, lib().muon_last_error().decode())


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _table(arr, dtype):
    if arr is None:
        return None, 0
    a = np.ascontiguousarray(arr)
    if a.dtype != dtype:
        a = np.ascontiguousarray(a.astype(dtype))
    return a, len(a)


def accumulate(accum, grad, scale: float, overwrite: bool = False, params=None, parts=None,
               n: int | None = None, stream=None):
    """accum += scale * bf16 grad (FP32), over parameter elements when tables
    are given, else over all n (= accum.numel()) elements."""
    p, np_ = _table(params, PARAM_DTYPE)
    q, nq = _table(parts, PART_DTYPE)
    if n is None:
        n = accum.numel() if hasattr(accum, "numel") else -1
    _check(lib().muon_accumulate(_ptr(accum), _ptr(grad), n, scale, int(overwrite),
                                 p.ctypes.data if p is not None else None, np_,
                                 q.ctypes.data if q is not None else None, nq, _stream(stream)))


ACCUMULATE_MAX = 8


def accumulate_n(accum, grads, scales, overwrite: bool = False, params=None, parts=None,
                 n: int | None = None, stream=None):
    """accumulate() over several micro-batches in one pass: the same bits as
    accumulate(accum, grads[j], scales[j], overwrite and j == 0) for j in
    order.  scales: one float for all, or one per micro-batch."""
    grads = list(grads)
    if not isinstance(scales, (list, tuple)):
        scales = [float(scales)] * len(grads)
    if len(scales) != len(grads):
        raise ValueError("one scale per micro-batch")
    p, np_ = _table(params, PARAM_DTYPE)
    q, nq = _table(parts, PART_DTYPE)
    if n is None:
        n = accum.numel() if hasattr(accum, "numel") else -1
    gp = (ctypes.c_void_p * max(len(grads), 1))(*[_ptr(g) for g in grads])
    sc = (ctypes.c_float * max(len(scales), 1))(*[float(x) for x in scales])
    _check(lib().muon_accumulate_n(_ptr(accum), ctypes.cast(gp, ctypes.c_void_p),
                                   ctypes.cast(sc, ctypes.c_void_p), len(grads), n, int(overwrite),
                                   p.ctypes.data if p is not None else None, np_,
                                   q.ctypes.data if q is not None else None, nq, _stream(stream)))


def step_options(clip_mode="update", grad_scale: float = 1.0, adam: dict | None = None,
                 workspace_budget: int = 0, last_grad=None, last_grad_scale: float = 1.0,
                 last_grad_overwrite: bool = False, stats_out=None, prev_grad=None,
                 prev_grad_scale: float = 1.0, prev_grad_overwrite: bool = False) -> StepOptions:
    """A muon_step_options_t.  adam: dict(lr, beta1, beta2, eps, step,
    exp_avg, exp_avg_sq) with device float buffers in accum's layout.
    last_grad: the last micro-batch's bf16 gradients (accum's layout), which
    the step accumulates itself, as accumulate(accum, last_grad,
    last_grad_scale, last_grad_overwrite) would (read by any of the step's
    kernels: keep it unchanged until the step is done).  stats_out: a device
    float64[4] the step fills with (sum of squares of the clip norm, skipped,
    NS problems, 0).  prev_grad: one more micro-batch folded in before
    last_grad (as accumulate(accum, prev_grad, prev_grad_scale,
    prev_grad_overwrite) would)."""
    o = StepOptions()
    o.struct_size = ctypes.sizeof(StepOptions)
    o.clip_mode = CLIP_MODES[clip_mode] if isinstance(clip_mode, str) else int(clip_mode)
    o.grad_scale = grad_scale
    o.workspace_budget = int(workspace_budget)
    if stats_out is not None:
        o.stats_out = _ptr(stats_out)
    if prev_grad is not None:
        o.prev_grad = _ptr(prev_grad)
        o.prev_grad_scale = prev_grad_scale
        o.prev_grad_overwrite = int(prev_grad_overwrite)
    if last_grad is not None:
        o.last_grad = _ptr(last_grad)
        o.last_grad_scale = last_grad_scale
        o.last_grad_overwrite = int(last_grad_overwrite)
    if adam is not None:
        o.aux_adam = 1
        o.adam_lr, o.adam_beta1 = adam["lr"], adam["beta1"]
        o.adam_beta2, o.adam_eps = adam["beta2"], adam["eps"]
        o.adam_step = int(adam["step"])
        o.exp_avg, o.exp_avg_sq = _ptr(adam["exp_avg"]), _ptr(adam["exp_avg_sq"])
    return o


def step(accum, momentum, master, params, parts, beta: float, lr: float, ns_method="gram",
         ns_steps: int = 5, clip: float = 0.0, operand_mode="bf16", result=None, stream=None,
         options: StepOptions | None = None):
    """One Muon step (overflow check, momentum, Newton-Schulz, global norm
    and clip, owned-slice write-back): muon_step, or muon_step_ex when
    `options` (see :func:`step_options`) is given.  Returns the device
    result buffer (torch int32[4]; decode with :func:`read_result`)."""
    import torch
    if result is None:
        result = torch.zeros(4, dtype=torch.int32, device=accum.device)
    p, np_ = _table(params, PARAM_DTYPE)
    q, nq = _table(parts, PART_DTYPE)
    method = NS_METHODS[ns_method] if isinstance(ns_method, str) else int(ns_method)
    mode = OPERAND_MODES[operand_mode] if isinstance(operand_mode, str) else int(operand_mode)
    args = (_ptr(accum), _ptr(momentum), _ptr(master), p.ctypes.data if np_ else None, np_,
            q.ctypes.data if nq else None, nq, beta, lr, method, ns_steps, clip, mode)
    if options is None:
        _check(lib().muon_step(*args, _ptr(result), _stream(stream)))
    else:
        _check(lib().muon_step_ex(*args, ctypes.byref(options), _ptr(result), _stream(stream)))
    return result


def step_ex(accum, momentum, master, params, parts, beta: float, lr: float, ns_method="gram",
            ns_steps: int = 5, clip: float = 0.0, operand_mode="bf16", clip_mode="update",
            grad_scale: float = 1.0, adam: dict | None = None, workspace_budget: int = 0,
            last_grad=None, last_grad_scale: float = 1.0, last_grad_overwrite: bool = False,
            prev_grad=None, prev_grad_scale: float = 1.0, prev_grad_overwrite: bool = False,
            stats_out=None, result=None, stream=None):
    """muon_step_ex with its options as keyword arguments."""
    return step(accum, momentum, master, params, parts, beta, lr, ns_method, ns_steps, clip,
                operand_mode, result, stream,
                step_options(clip_mode, grad_scale, adam, workspace_budget, last_grad,
                             last_grad_scale, last_grad_overwrite, stats_out, prev_grad,
                             prev_grad_scale, prev_grad_overwrite))


def describe_tables(params, parts, ns_method="gram", operand_mode="bf16") -> dict:
    """muon_describe_tables: what a step over these tables would do, on the
    host alone (validation, block and stacking counts, workspace size)."""
    p, np_ = _table(params, PARAM_DTYPE)
    q, nq = _table(parts, PART_DTYPE)
    method = NS_METHODS[ns_method] if isinstance(ns_method, str) else int(ns_method)
    mode = OPERAND_MODES[operand_mode] if isinstance(operand_mode, str) else int(operand_mode)
    info = TableInfo()
    _check(lib().muon_describe_tables(p.ctypes.data if np_ else None, np_,
                                      q.ctypes.data if nq else None, nq, method, mode,
                                      ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in TableInfo._fields_}


def read_result(result) -> dict:
    """Decode the 16-byte device result struct (synchronises on the copy)."""
    r = result.cpu().numpy().astype(np.int32)
    f = r.view(np.float32)
    return {"applied": int(r[0]), "ns_calls": int(r[1]),
            "global_norm": float(f[2]), "clip_coef": float(f[3])}


def newton_schulz(X, Y=None, ns_method="gram", ns_steps: int = 5, operand_mode="bf16",
                  stream=None):
    """Orthogonalise one matrix X (bf16 or fp32, rows x cols) into Y."""
    import torch
    if X.dim() != 2:
        raise ValueError("X must be 2-D")
    if Y is None:
        Y = torch.empty_like(X)
    io = {torch.bfloat16: 0, torch.float32: 1}[X.dtype]
    if Y.dtype != X.dtype or Y.shape != X.shape:
        raise ValueError("Y must match X's shape and dtype")
    method = NS_METHODS[ns_method] if isinstance(ns_method, str) else int(ns_method)
    mode = OPERAND_MODES[operand_mode] if isinstance(operand_mode, str) else int(operand_mode)
    _check(lib().muon_newton_schulz(_ptr(X), _ptr(Y), X.shape[0], X.shape[1], io, method,
                                    ns_steps, mode, _stream(stream)))
    return Y


def get_stats() -> dict:
    s = Stats()
    _check(lib().muon_get_stats(ctypes.byref(s)))
    return {k: getattr(s, k) for k, _ in Stats._fields_}


def last_error() -> str:
    return lib().muon_last_error().decode()


def release_workspace():
    lib().muon_release_workspace()


def device_error() -> int:
    return int(lib().muon_device_error())


def profile_enable(on: bool = True, phases=None):
    """Time every phase (on), none, or only `phases` (names from PHASES)."""
    if phases is None:
        _check(lib().muon_profile_enable(int(on)))
    else:
        mask = 0
        for name in phases:
            mask |= 1 << PHASES.index(name)
        _check(lib().muon_profile_enable_phases(mask if on else 0))


def profile_read(reset: bool = False) -> dict:
    arr = (PhaseTime * len(PHASES))()
    _check(lib().muon_profile_read(arr, len(PHASES), int(reset)))
    return {name: {"launches": arr[i].launches, "ms": arr[i].total_ms,
                   "bytes": arr[i].algorithmic_bytes, "flops": arr[i].algorithmic_flops}
            for i, name in enumerate(PHASES)}


# muon_testing_set knobs and their product-path defaults
TEST_KNOBS = {"gemm": (0, 0), "stack": (1, 1), "flow": (2, 1), "flow_lag": (3, 0),
              "flow_waves": (4, 1), "raster": (5, 0), "extent_shrink": (6, 0)}
TEST_GEMM = {"default": 0, "simt": 1, "tc1": 2}


class testing:
    """Cross-check context for tests: plans built inside it route the
    Newton-Schulz products as the knobs say (gemm="simt" CUDA-core GEMM,
    gemm="tc1" single-SM tensor-core kernel, stack=0, flow=0, flow_lag=k,
    flow_waves=k, raster=1 row-major tile order).  Plans are dropped on entry and exit, and every knob
    returns to its product-path default on exit."""

    def __init__(self, **knobs):
        self.knobs = knobs

    def __enter__(self):
        release_workspace()
        for name, value in self.knobs.items():
            if name == "gemm" and isinstance(value, str):
                value = TEST_GEMM[value]
            _check(lib().muon_testing_set(TEST_KNOBS[name][0], int(value)))
        return self

    def __exit__(self, *exc):
        release_workspace()
        for knob, default in TEST_KNOBS.values():
            _check(lib().muon_testing_set(knob, default))
        return False
