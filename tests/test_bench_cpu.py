"""The bench's reference arm runs on the host alone (the oracle timed on a
bounded sample of the Llama-3-8B step, extrapolated by formula flops) and
prints the contract's single JSON line, whose fields say what was timed."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--cpu-budget", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "ms" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["value"] == d["cpu_baseline"]["value"]
    assert d["steps"] == 1 and d["warmup"] == 3
    # a sampled arm: ms_per_step is the time of one timed (sample) step, and
    # the value is that time scaled to the whole step
    assert d["sampled"] is True and d["sample_scale"] > 1
    assert abs(d["value"] - d["ms_per_step"] * d["sample_scale"]) <= 1e-6 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["cpu"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_roofline_traffic_records_match_the_sources():
    """The DRAM traffic the bench reports beside its roofline comes from ncu
    captures of particular sources; a record whose kernel or task order has
    changed since reads as null in the bench line.  The records for the
    headline (Llama-3-8B), GPT-2-small and ragged workloads must match the
    sources as committed."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.gemm_traffic("llama") is not None
    assert bench.gemm_traffic("gpt2") is not None
    assert bench._traffic_if_current(bench.RAGGED_NS_TRAFFIC, "bytes_per_step") is not None


def test_sweep_and_ragged_cpu_baselines_say_what_was_timed(monkeypatch):
    """The oracle baselines of the sweep and ragged lines: a shape within
    the full-timing bound is timed whole; a larger one is the bound's square
    scaled by formula flops; the ragged step is timed on a prefix of the
    matrices and scaled by gram flops, or whole when the budget allows."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import workloads as wl
    monkeypatch.setattr(bench, "SWEEP_CPU_FULL_MAX", 32)
    cache = {}
    whole = bench.sweep_cpu_baseline(32, 24, "standard", "bf16", cache)
    assert whole["sampled"] is False and whole["value"] > 0 and whole["kind"] == "oracle"
    big = bench.sweep_cpu_baseline(64, 128, "gram", "fp32", cache)
    ratio = (4.0 * 64 * 64 * 128 + 34.0 * 64 ** 3) / (4.0 * 32 ** 3 + 34.0 * 32 ** 3)
    assert big["sampled"] is True and ("gram", "fp32") in cache
    assert abs(big["value"] - 1000.0 * cache[("gram", "fp32")] * ratio) <= 1e-9 * big["value"]
    lay = wl.ragged_layout(160, seed=7)
    mats = [wl.rng_for(7, 2, i).standard_normal((s.rows, s.cols), dtype=np.float32)
            for i, s in enumerate(lay.specs)]
    part = bench.ragged_cpu_baseline(lay, mats, "bf16", 0.0)
    assert part["sampled"] is True and "first 128 of 160" in part["sample"]
    full = bench.ragged_cpu_baseline(lay, mats, "bf16", 1e9)
    assert full["sampled"] is False and "first 160 of 160" in full["sample"]
    assert abs(full["value"] - 1000.0 * full["sample_seconds"]) <= 1e-9 * full["value"]
