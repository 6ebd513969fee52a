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
