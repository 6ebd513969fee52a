"""The library's host planner, without a GPU (muon_describe_tables): table
validation, per-head blocks, the stacking of equal consecutive head blocks,
partition cuts and the unbounded workspace, each against an expectation
derived here from the shapes alone."""
import numpy as np
import pytest

import newton_schulz_fp32_gb300 as nsg
import workloads as wl


@pytest.fixture(scope="module")
def lib():
    nsg.build()
    return nsg.lib()


def round_up(x, a):
    return (x + a - 1) // a * a


def cut_segments(layout, heads_of):
    """(block or auxiliary parameter) x partition runs, counted from the
    flat ranges: a block is one run plus one per partition boundary strictly
    inside it."""
    bounds = sorted({int(q["flat_begin"]) for q in layout.parts} |
                    {int(q["flat_end"]) for q in layout.parts})
    n = 0
    for spec, row in zip(layout.specs, layout.params):
        h = max(1, heads_of(spec))
        step = spec.numel // h
        for b in range(h):
            lo = int(row["offset"]) + b * step
            hi = lo + step
            n += 1 + sum(1 for x in bounds if lo < x < hi)
    return n


def test_tiny_config(lib):
    # 17x13 and 9x17 Muon matrices, an 8x5 auxiliary group; each group its
    # own 16 x 2-aligned segment cut in two (17x13 at [0,221), pad 3; 9x17
    # at [224,377), pad 7; 8x5 at [384,424), pad 24)
    d = nsg.describe_tables(wl.tiny_layout().params, wl.tiny_layout().parts, "standard", "fp32")
    assert d["muon_params"] == 2 and d["muon_blocks"] == 2 and d["ns_problems"] == 2
    assert d["muon_elements"] == 17 * 13 + 9 * 17 and d["aux_elements"] == 40
    assert d["padding_elements"] == 3 + 7 + 24
    assert d["segments"] == 6
    assert d["pair_engine"] == 0 and d["stack_rows"] == 128   # blocks far below 192 rows


@pytest.mark.parametrize("method,operand,x_bytes,sq_planes,sq_bytes",
                         [("standard", "bf16", 2, 2, 2), ("gram", "bf16", 2, 5, 6),
                          ("standard", "fp32", 6, 2, 6), ("gram", "fp32", 6, 5, 6)])
def test_gpt2_small_plan(lib, method, operand, x_bytes, sq_planes, sq_bytes):
    lay = wl.gpt2_small_layout()
    d = nsg.describe_tables(lay.params, lay.parts, method, operand)
    # 12 layers x (Q, K with 12 heads of 64 rows; V, O; MLP up, down)
    assert d["muon_params"] == 72 and d["muon_blocks"] == 12 * (12 + 12 + 4)
    # Q and K heads (64-row blocks, a multiple of 32, adjacent and equal)
    # stack into problems of the engine's row tile: four into 256 rows on SM
    # pairs (standard form, BF16 operands: every problem then at least 192
    # rows), two into 128 rows on single SMs (split-3 FP32, and the gram
    # form, whose m x m recurrence grows with the stack); plus V, O, up, down
    per = 4 if (operand == "bf16" and method == "standard") else 2
    assert d["ns_problems"] == 12 * (2 * 12 // per + 4)
    assert d["pair_engine"] == (1 if per == 4 else 0)
    assert d["stack_rows"] == 64 * per
    assert d["muon_elements"] == 12 * (4 * 768 * 768 + 2 * 3072 * 768) and d["aux_elements"] == 0
    assert d["padding_elements"] == 0          # 84,934,656 is a multiple of 128 x 8
    assert d["segments"] == cut_segments(lay, lambda s: s.num_heads)
    # work regions: two m x n X regions over all blocks (m <= n, rows padded
    # to 8 elements, regions to 64), and the m x m regions per problem
    x = 12 * (24 * round_up(64 * 768, 64) + 2 * 768 * 768 + 2 * 768 * 3072)
    sq = 12 * (2 * 12 // per * (64 * per) ** 2 + 4 * 768 * 768)
    assert d["workspace_bytes"] == 2 * x_bytes * x + sq_planes * sq_bytes * sq + 256


def test_llama3_8b_plan(lib):
    lay = wl.build_layout([wl.llama3_8b_specs()], 128, 64)
    d = nsg.describe_tables(lay.params, lay.parts, "standard", "bf16")
    assert d["muon_blocks"] == 32 * 7 and d["ns_problems"] == 32 * 7   # nothing to stack
    assert d["pair_engine"] == 1
    per_layer = 2 * 4096 * 4096 + 2 * 1024 * 4096 + 3 * 14336 * 4096
    assert d["muon_elements"] == 32 * per_layer
    assert d["segments"] == cut_segments(lay, lambda s: 1)
    # m x m regions: Q, O 4096, K, V 1024, gate, up, down 4096
    x = 32 * per_layer
    sq = 32 * (5 * 4096 * 4096 + 2 * 1024 * 1024)
    assert d["workspace_bytes"] == 2 * 2 * x + 2 * 2 * sq + 256


def test_ragged_blocks_use_single_sms(lib):
    lay = wl.ragged_layout(512, seed=1003)
    d = nsg.describe_tables(lay.params, lay.parts, "gram", "bf16")
    assert d["muon_blocks"] == 512 and d["pair_engine"] == 0 and d["stack_rows"] == 128
    assert d["ns_problems"] <= 512


def test_ragged_blocks_stack_by_shape(lib):
    """Randomly ordered small matrices stack as if grouped by shape: per
    canonical shape (m, n), blocks of 32 or 64 rows fill 128-row stacks."""
    from collections import Counter
    lay = wl.ragged_layout(2048, seed=1003)
    shapes = Counter((min(s.rows, s.cols), max(s.rows, s.cols)) for s in lay.specs)
    want = sum(-(-c // (128 // m)) if m % 32 == 0 and 2 * m <= 128 else c
               for (m, n), c in shapes.items())
    d = nsg.describe_tables(lay.params, lay.parts, "gram", "bf16")
    assert d["ns_problems"] == want < 2048


def test_describe_rejects_what_the_step_rejects(lib):
    bad = np.zeros(1, dtype=nsg.PARAM_DTYPE)
    bad[0] = (0, 10, 8, 3, 1)                        # 10 rows in 3 heads
    parts = np.zeros(1, dtype=nsg.PART_DTYPE)
    parts[0] = (0, 80, 0)
    with pytest.raises(nsg.MuonError):
        nsg.describe_tables(bad, parts)
    assert "heads" in lib.muon_last_error().decode() or "num_heads" in lib.muon_last_error().decode()
    with pytest.raises(nsg.MuonError):
        nsg.describe_tables(wl.tiny_layout().params, wl.tiny_layout().parts, 7, "bf16")


def test_auxiliary_only_and_empty_tables(lib):
    lay = wl.build_layout([[wl.ParamSpec("ln", 1, 768, use_muon=False),
                            wl.ParamSpec("emb", 40, 96, use_muon=False)]], 128, 2)
    d = nsg.describe_tables(lay.params, lay.parts)
    assert d["muon_params"] == d["muon_blocks"] == d["ns_problems"] == 0
    assert d["aux_elements"] == 768 + 40 * 96 and d["workspace_bytes"] == 0
    total = int(sum(int(q["flat_end"]) - int(q["flat_begin"]) for q in lay.parts))
    assert d["padding_elements"] == total - 768 - 40 * 96
    e = nsg.describe_tables([], [])   # (the engine choice is vacuous without blocks)
    assert all(v == 0 for k, v in e.items() if k not in ("stack_rows", "pair_engine"))
