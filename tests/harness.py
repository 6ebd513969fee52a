"""Helpers shared by the GPU parity tests: seeded inputs on both sides, the
library call through the C ABI (Python binding), and comparison rules.

Tolerances (written here once, used by every parity test):
* bit-exact: accumulation, momentum, ownership, padding, overflow skips,
  partition independence -- integer-like bookkeeping and FP32 element
  arithmetic done in the same order on both sides;
* BF16 operand mode: per matrix, relative Frobenius error <= 1e-2 against
  the oracle's bf16-emulating mode;
* FP32 operand mode: atol 1e-4 / rtol 1e-3 against the oracle's exact
  (fp64) mode -- the tolerance of the pages' compiled-NS check ("Support
  Muon in BF16_Optimizer with FP32 gradient accumulation", validation
  table)."""
import numpy as np

import workloads as wl

BF16_RELF = 1e-2
FP32_ATOL, FP32_RTOL = 1e-4, 1e-3
ORACLE_MODE = {"bf16": "bf16", "fp32": "exact"}


def relf(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def assert_close_update(got, want, mode, what=""):
    """Compare one matrix's NS update by the operand mode's rule."""
    if mode == "bf16":
        e = relf(got, want)
        assert e <= BF16_RELF, f"{what}: rel-F {e:.3e} > {BF16_RELF}"
    else:
        got = np.asarray(got, np.float64)
        want = np.asarray(want, np.float64)
        bad = np.abs(got - want) > FP32_ATOL + FP32_RTOL * np.abs(want)
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside atol/rtol, max err "
                               f"{np.abs(got - want).max():.3e}")


def bits(x):
    return np.ascontiguousarray(x, np.float32).view(np.uint32)


def to_dev(x, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_tensor(bits_u16, torch):
    """uint16 bit patterns -> a device bfloat16 tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).cuda().view(torch.bfloat16)


class GpuState:
    """accum / momentum / master storage buffers on the device."""

    def __init__(self, torch, accum, momentum, master):
        self.torch = torch
        self.accum = to_dev(accum, torch)
        self.momentum = to_dev(momentum, torch)
        self.master = to_dev(master, torch)

    def numpy(self):
        return (self.accum.cpu().numpy(), self.momentum.cpu().numpy(), self.master.cpu().numpy())


def micro_batch_grads(layout, seed, step, gas, sigmas=None):
    """Per-parameter bf16-valued gradients of each micro-batch of a step."""
    return [wl.gaussian_grads(layout, seed, step * gas + mb, sigmas) for mb in range(gas)]
