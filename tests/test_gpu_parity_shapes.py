"""Newton-Schulz entry against the oracle at the sweep's mid sizes and in
both orientations of one matrix.

* 2048^2 and 4096^2 (the sweep's sizes the host oracle still finishes in
  seconds), standard and gram, BF16 and FP32 operands, element by element
  by the operand mode's rule (BF16: rel-F <= 1e-2 against the
  BF16-emulating oracle; FP32: atol 1e-4 / rtol 1e-3 against the exact
  oracle, the tolerance of the compiled-NS check in "Support Muon in
  BF16_Optimizer with FP32 gradient accumulation", validation table).
* Transpose equivariance: NS(X^T) = NS(X)^T bit for bit.  A tall input is
  transposed into the same canonical m x n problem as its wide transpose,
  so every product is the same; only the order in which the normalising
  sum of squares is taken differs, which moves the FP32 divisor only when
  the double sum sits at an FP32 rounding boundary."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl
from harness import ORACLE_MODE, assert_close_update, bits, to_dev
from oracle import newton_schulz as ons

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    nsg.build()
    return t


def device_input(torch, G, mode):
    if mode == "bf16":
        return to_dev(G, torch, torch.bfloat16)
    return to_dev(G, torch)


def host_input(shape, mode, seed):
    G = wl.rng_for(seed, *shape).standard_normal(shape).astype(np.float32)
    return wl.to_bf16_values(G) if mode == "bf16" else G


@pytest.mark.parametrize("n", [2048, 4096])
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_sweep_mid_sizes_against_oracle(torch, n, method, mode):
    G = host_input((n, n), mode, wl.CONFIG_SEED["sweep"] + n)
    Y = nsg.newton_schulz(device_input(torch, G, mode), ns_method=method, ns_steps=5,
                          operand_mode=mode)
    got = Y.float().cpu().numpy()
    want = ons.newton_schulz(G, method, 5, ORACLE_MODE[mode])
    assert_close_update(got, want, mode, f"{n}^2 {method} {mode}")
    nsg.release_workspace()
    assert nsg.device_error() == 0


@pytest.mark.parametrize("shape", [(77, 300), (1000, 1500)])
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_transpose_equivariance_bitwise(torch, shape, method, mode):
    G = host_input(shape, mode, 53)
    wide = nsg.newton_schulz(device_input(torch, G, mode), ns_method=method,
                             operand_mode=mode).float().cpu().numpy()
    tall = nsg.newton_schulz(device_input(torch, G.T.copy(), mode), ns_method=method,
                             operand_mode=mode).float().cpu().numpy()
    assert np.array_equal(bits(tall), bits(wide.T.copy())), f"{shape} {method} {mode}"
    # and the pair against the oracle
    assert_close_update(wide, ons.newton_schulz(G, method, 5, ORACLE_MODE[mode]), mode,
                        f"{shape} {method} {mode} vs oracle")
    assert nsg.device_error() == 0
