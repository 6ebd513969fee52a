"""Benchmark of the Muon optimizer step on GB300.

Default workload (the benchmark line): the Llama-3-8B-shaped parameter set
(32 layers of Q, O 4096x4096, K, V 1024x4096, gate, up 14336x4096, down
4096x14336; 6.98G elements, 64 partitions, 128 alignment; even-indexed
matrices rank 8 plus 1e-3 noise, odd-indexed N(0,1)), two BF16 micro-batches
accumulated in FP32, then one Muon step (5 standard Newton-Schulz steps,
BF16 operands).  One timed step = one muon_step_ex that accumulates both
micro-batches itself (options prev_grad and last_grad: they overwrite accum,
so the step forms the gradient from them wherever it reads it), all
kernels of the library, every input resident in HBM (accum, momentum and master
are 27.9 GB each, far larger than the 129 MB L2, so no flush is needed);
the K timed steps are recorded into one CUDA graph and timed as one replay.
``--workload gpt2`` runs the same contract line on the GPT-2-small
parameter set (84.9M elements, P=8, four micro-batches, clip 0.05), which
the default line also summarises.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "Muon step time & NS TFLOP/s (% of GB300 bf16 dense peak) plus HBM GB/s, 1 GPU"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch of the BF16 pair GEMM (one launch runs all NS
# products of a step), from ncu (dram__bytes_read.sum +
# dram__bytes_write.sum, averaged over two launches), valid only for the
# sources they were taken on (hash below: the kernel, and for Llama-3-8B
# also the planner whose task order sets the L2 reuse).  GPT-2: the full
# step.  Llama-3-8B: the full step is too large to capture, so one layer
# (the same seven shapes) was captured, 13.136 GB per launch, and scaled by
# the 32 layers.
GEMM_TRAFFIC = {
    "gpt2": {"bytes_per_launch": 3.8480e9, "sources_sha256_16": "7179c2b5092211c5",
             "files": ["newton_schulz_fp32_gb300/csrc/gemm_tc2.cu",
                       "newton_schulz_fp32_gb300/csrc/tc_common.cuh"]},
    "llama": {"bytes_per_launch": 32 * 13.1362e9, "sources_sha256_16": "932fe30ce6969503",
              "files": ["newton_schulz_fp32_gb300/csrc/gemm_tc2.cu",
                        "newton_schulz_fp32_gb300/csrc/tc_common.cuh",
                        "newton_schulz_fp32_gb300/csrc/api.cu"]},
}


# DRAM bytes of the ragged gram step's 16 GEMM launches (R0, the 14 launches
# of the split-3 m x m recurrence, Y), summed from one ncu capture of the
# full 8192-matrix step (dram__bytes_read.sum + dram__bytes_write.sum,
# one pass), valid for the sources hashed.
RAGGED_NS_TRAFFIC = {"bytes_per_step": 46.476e9, "sources_sha256_16": "5bd3eca0ff84a1f3",
                     "files": ["newton_schulz_fp32_gb300/csrc/gemm_tc3.cu",
                               "newton_schulz_fp32_gb300/csrc/gemm_tc.cu",
                               "newton_schulz_fp32_gb300/csrc/tc_common.cuh",
                               "newton_schulz_fp32_gb300/csrc/api.cu"]}


def _traffic_if_current(rec, key):
    import hashlib
    h = hashlib.sha256()
    for f in rec["files"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return rec[key] if h.hexdigest()[:16] == rec["sources_sha256_16"] else None


def gemm_traffic(workload):
    import hashlib
    rec = GEMM_TRAFFIC.get(workload)
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in rec["files"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != rec["sources_sha256_16"]:
        return None   # the kernel or its task order changed since the counters were taken
    return rec["bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def peak_value(peaks, key):
    for k in (key, key.replace("_gbs", "_GBps")):
        if k in peaks and isinstance(peaks[k], (int, float)):
            return float(peaks[k])
    return FALLBACK[key]


# ------------------------------------------------------------------ workloads

class Workload:
    """One benchmark configuration: its layout, micro-batch count and step
    settings, and how its device and pinned host inputs are made."""

    def __init__(self, name, lay, gas, ns_method, clip, desc):
        self.name, self.lay, self.gas = name, lay, gas
        self.ns_method, self.clip, self.desc = ns_method, clip, desc


def gpt2_workload(ns_method, mode):
    lay = wl.gpt2_small_layout()
    desc = (f"gpt2-small muon step: 12 layers (q,k 12-head, v, o 768x768; up 3072x768; "
            f"down 768x3072), 84.9M params, P=8, align 128, gas=4 bf16 grads, "
            f"{ns_method} NS x5, {mode} operands, clip 0.05; the four micro-batches are "
            f"accumulated in one pass (muon_accumulate_n)")
    return Workload("gpt2", lay, 4, ns_method, 0.05, desc)


def llama_workload(mode, layers=32):
    lay = wl.llama3_8b_layout(layers=layers)
    desc = (f"llama3-8b muon step: {layers} layers (q,o 4096x4096; k,v 1024x4096; gate,up "
            f"14336x4096; down 4096x14336), {lay.n_param_elements / 1e9:.2f}G params, P=64, "
            f"align 128, gas=2 bf16 grads (even-indexed matrices rank 8 + 1e-3 noise), "
            f"standard NS x5, {mode} operands; both micro-batches are accumulated inside "
            f"the step")
    return Workload("llama", lay, 2, "standard", 0.0, desc)


def make_inputs(torch, W, stream, host_copies=True):
    """Device state and micro-batch gradients, plus pinned host copies of the
    gradients (the end-to-end run copies them in every step)."""
    lay = W.lay
    n = lay.storage_size
    with torch.cuda.stream(stream):
        if W.name == "gpt2":
            seed = wl.CONFIG_SEED["gpt2"]
            sig = wl.loguniform_sigmas(lay, seed, 1e-4, 1e-1)
            grads = [wl.bf16_storage_grad(lay, wl.gaussian_grads(lay, seed, mb, sig))
                     for mb in range(W.gas)]
            m0 = wl.pack(lay, [0.1 * g for g in wl.gaussian_grads(lay, seed, 100, sig, bf16=False)])
            w0 = wl.pack(lay, wl.gaussian_grads(lay, seed, 101, None, bf16=False))
            acc = torch.zeros(n, dtype=torch.float32, device="cuda")
            mom = torch.from_numpy(m0).cuda()
            mst = torch.from_numpy(w0).cuda()
            g_dev = [torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16) for g in grads]
        else:
            seed = wl.CONFIG_SEED["llama"]
            gen = torch.Generator(device="cuda").manual_seed(seed)
            acc = torch.zeros(n, dtype=torch.float32, device="cuda")
            mom = torch.zeros(n, dtype=torch.float32, device="cuda")
            mst = torch.randn(n, dtype=torch.float32, device="cuda", generator=gen)
            g_dev = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(W.gas)]
            for mb in range(W.gas):
                wl.llama_grad_into(lay, seed, mb, g_dev[mb])
        g_host = []
        if host_copies:
            g_host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(W.gas)]
            for h, d in zip(g_host, g_dev):
                h.copy_(d)
    torch.cuda.synchronize()
    return acc, mom, mst, g_dev, g_host


def ns_formula_flops(lay, method, steps=5):
    """Algorithmic Newton-Schulz flops of one step: standard 5(4m^2n+2m^3),
    gram 4m^2n + 34m^3 (5 steps), per head block."""
    f = 0.0
    for s in lay.specs:
        if not s.use_muon:
            continue
        h = s.num_heads if s.num_heads > 1 else 1
        r, c = s.rows // h, s.cols
        m, n = min(r, c), max(r, c)
        if method == "standard":
            f += h * steps * (4.0 * m * m * n + 2.0 * m ** 3)
        else:
            f += h * (4.0 * m * m * n + (2 * steps + 2 * (steps - 1) + 4 * (steps - 1)) * m ** 3)
    return f


def ns_executed_flops_pairs(lay, steps=5, tile=256):
    """Flops the SM-pair kernel executes for the standard form in BF16 mode:
    X X^T and c A^2 + b A compute only the 256x256 tiles touching the upper
    triangle (mirrored), X' = B X + a X every tile.  Counted per NS problem
    (unstacked blocks of 192+ rows)."""
    f = 0.0
    for s in lay.specs:
        if not s.use_muon:
            continue
        h = s.num_heads if s.num_heads > 1 else 1
        r, c = s.rows // h, s.cols
        m, n = min(r, c), max(r, c)
        nt = -(-m // tile)
        sym = nt * (nt + 1) // 2 * tile * tile
        f += h * steps * (2.0 * sym * n + 2.0 * sym * m + 2.0 * m * m * n)
    return f


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing

def cpu_info():
    """(threads the oracle's BLAS may use, CPU model string)."""
    cores = os.cpu_count() or 1
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            cores = int(os.environ[var])
            break
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return cores, model


def _oracle_mode(mode):
    return "bf16" if mode == "bf16" else "exact"


def oracle_step_gpt2(ns_method, mode):
    """The oracle's whole GPT-2-small step (accumulate x4, momentum, NS, norm,
    clip, write-back over all 12 layers, P=8); returns seconds."""
    import oracle.muon as om
    import oracle.bf16 as obf
    lay = wl.gpt2_small_layout()
    seed = wl.CONFIG_SEED["gpt2"]
    sig = wl.loguniform_sigmas(lay, seed, 1e-4, 1e-1)
    grads = [obf.bits_to_f32(wl.bf16_storage_grad(lay, wl.gaussian_grads(lay, seed, mb, sig)))
             for mb in range(4)]
    m0 = wl.pack(lay, [0.1 * g for g in wl.gaussian_grads(lay, seed, 100, sig, bf16=False)])
    w0 = wl.pack(lay, wl.gaussian_grads(lay, seed, 101, None, bf16=False))
    t0 = time.perf_counter()
    acc = None
    for mb in range(4):
        acc = om.accumulate(acc, grads[mb], 0.25, overwrite=(mb == 0))
    om.muon_step_flat(acc, m0, w0, lay.params, lay.parts, 0.95, 0.02, ns_method, 5, 0.05,
                      _oracle_mode(mode))
    return time.perf_counter() - t0


# Llama-3-8B matrices in the order the bounded sample takes them (layer 0:
# k, v, o, q, then gate, up, down): the smallest first, so a short budget
# still times whole matrices.
LLAMA_SAMPLE_ORDER = [1, 2, 3, 0, 4, 5, 6]


def oracle_step_llama_sample(mode, budget_s):
    """The oracle's whole step (accumulate x2, momentum, NS, norm, write-back)
    on layer-0 matrices of the Llama-3-8B set, one matrix at a time in
    LLAMA_SAMPLE_ORDER until budget_s is spent (at least one).  Inputs are
    numpy-seeded with the workload's distribution (even-indexed matrices rank
    8 + 1e-3 noise, odd-indexed N(0,1), bf16).  Returns (seconds, formula
    flops of the matrices timed, their names)."""
    import oracle.muon as om
    full = wl.llama3_8b_layout(layers=1)
    seed = wl.CONFIG_SEED["llama"]
    spent, flops, names = 0.0, 0.0, []
    for k in LLAMA_SAMPLE_ORDER:
        spec = full.specs[k]
        lay = wl.build_layout([[spec]], 128, 1)
        mats = []
        for mb in range(2):
            rng = wl.rng_for(seed, 7, k, mb)
            if k % 2 == 0:
                g = (rng.standard_normal((spec.rows, 8), dtype=np.float32)
                     @ rng.standard_normal((8, spec.cols), dtype=np.float32)
                     + np.float32(1e-3) * rng.standard_normal((spec.rows, spec.cols), dtype=np.float32))
            else:
                g = rng.standard_normal((spec.rows, spec.cols), dtype=np.float32)
            mats.append(wl.pack(lay, [wl.to_bf16_values(g)]))
        z = np.zeros(lay.storage_size, np.float32)
        t0 = time.perf_counter()
        acc = om.accumulate(None, mats[0], 0.5, overwrite=True)
        acc = om.accumulate(acc, mats[1], 0.5)
        om.muon_step_flat(acc, z, z, lay.params, lay.parts, 0.95, 0.02, "standard", 5, 0.0,
                          _oracle_mode(mode))
        spent += time.perf_counter() - t0
        flops += ns_formula_flops(lay, "standard")
        names.append(f"{spec.name} {spec.rows}x{spec.cols}")
        if spent >= budget_s:
            break
    return spent, flops, names


def cpu_baseline(workload, ns_method, mode, budget_s):
    """The oracle timed on the host cores: GPT-2-small in full (one rep), or
    a bounded sample of the Llama-3-8B step extrapolated by formula flops.
    Returns the contract's cpu_baseline object (value in ms per full step)."""
    cores, model = cpu_info()
    if workload == "gpt2":
        sec = oracle_step_gpt2(ns_method, mode)
        return {"value": 1000.0 * sec, "unit": "ms", "cores": cores, "cpu": model,
                "kind": "oracle", "sampled": False,
                "sample": f"oracle ({_oracle_mode(mode)} mode, numpy fp64 BLAS) on the whole "
                          f"GPT-2-small step (12 layers, P=8), one rep"}
    sec, flops, names = oracle_step_llama_sample(mode, budget_s)
    total = ns_formula_flops(wl.llama3_8b_layout(), "standard")
    return {"value": 1000.0 * sec * total / flops, "unit": "ms", "cores": cores, "cpu": model,
            "kind": "oracle", "sampled": True, "sample_seconds": sec,
            "sample_fraction_of_step_flops": flops / total,
            "sample": f"oracle ({_oracle_mode(mode)} mode, numpy fp64 BLAS) on the whole step of "
                      f"{len(names)} layer-0 matrices ({', '.join(names)}) in {sec:.1f} s, "
                      f"extrapolated to the 224-matrix step by formula flops "
                      f"(x{total / flops:.0f})"}


SWEEP_CPU_FULL_MAX = 4096   # sweep shapes up to this size are timed in full on the host


def sweep_cpu_baseline(r, c, ns_method, mode, cache):
    """The oracle's Newton-Schulz of one r x c matrix (N(0,1), bf16-valued in
    BF16 mode) on the host cores: timed in full up to 4096 on each side,
    else the 4096 x 4096 time scaled by formula flops (cached per method and
    mode)."""
    import oracle.newton_schulz as ons
    import oracle.bf16 as obf
    cores, model = cpu_info()

    def flops(rr, cc):
        m, n = min(rr, cc), max(rr, cc)
        return 5 * (4.0 * m * m * n + 2.0 * m ** 3) if ns_method == "standard" \
            else 4.0 * m * m * n + 34.0 * m ** 3

    def run(rr, cc):
        rng = wl.rng_for(wl.CONFIG_SEED["sweep"], rr, cc)
        X = rng.standard_normal((rr, cc), dtype=np.float32)
        if mode == "bf16":
            X = obf.round_bf16(X)
        t0 = time.perf_counter()
        ons.newton_schulz(X, ns_method, 5, _oracle_mode(mode))
        return time.perf_counter() - t0

    base = {"unit": "ms", "cores": cores, "cpu": model, "kind": "oracle"}
    if max(r, c) <= SWEEP_CPU_FULL_MAX:
        sec = run(r, c)
        return dict(base, value=1000.0 * sec, sampled=False,
                    sample=f"oracle ({_oracle_mode(mode)} mode, numpy fp64 BLAS) on the whole "
                           f"{r}x{c} Newton-Schulz, one rep")
    key = (ns_method, mode)
    if key not in cache:
        cache[key] = run(SWEEP_CPU_FULL_MAX, SWEEP_CPU_FULL_MAX)
    sec = cache[key]
    scale = flops(r, c) / flops(SWEEP_CPU_FULL_MAX, SWEEP_CPU_FULL_MAX)
    return dict(base, value=1000.0 * sec * scale, sampled=True, sample_seconds=sec,
                sample=f"oracle ({_oracle_mode(mode)} mode) on a {SWEEP_CPU_FULL_MAX}x"
                       f"{SWEEP_CPU_FULL_MAX} matrix in {sec:.1f} s, scaled to {r}x{c} by "
                       f"formula flops (x{scale:.1f})")


def ragged_cpu_baseline(lay, mats, mode, budget_s):
    """The oracle's whole gram Muon step on the first matrices of the ragged
    set (momentum, norm, Newton-Schulz, write-back), as many as about
    budget_s of host time allows, extrapolated to all of them by gram
    formula flops."""
    import oracle.muon as om
    cores, model = cpu_info()
    total = ns_formula_flops(lay, "gram")
    k, sec, done = 128, 0.0, 0
    while True:
        sub = wl.build_layout([lay.specs[:k]], 128, 1)
        g = wl.pack(sub, mats[:k])
        z = np.zeros_like(g)
        t0 = time.perf_counter()
        om.muon_step_flat(g, z, z.copy(), sub.params, sub.parts, 0.95, 0.02, "gram", 5, 0.0,
                          _oracle_mode(mode))
        sec, done = time.perf_counter() - t0, k
        if k >= len(lay.specs) or sec * 4 > budget_s:
            break
        k = min(4 * k, len(lay.specs))
    part = ns_formula_flops(wl.build_layout([lay.specs[:done]], 128, 1), "gram")
    full = done >= len(lay.specs)
    return {"value": 1000.0 * sec * total / part, "unit": "ms", "cores": cores, "cpu": model,
            "kind": "oracle", "sampled": not full, "sample_seconds": sec,
            "sample": f"oracle ({_oracle_mode(mode)} mode, numpy fp64 BLAS) on the whole gram "
                      f"step of the first {done} of {len(lay.specs)} matrices in {sec:.1f} s"
                      + ("" if full else f", extrapolated by gram formula flops "
                                         f"(x{total / part:.1f})")}


# ------------------------------------------------------------------ GPU run

def run_gpu(args, W, rank, world):
    """One GPU, all partitions emulated on it: warm-up, the K timed steps as
    one CUDA-graph replay (inputs resident), an eager pass of the same steps
    for the phase split, and the end-to-end loop with host copies.  Returns
    a dict of measurements."""
    import torch
    import newton_schulz_fp32_gb300 as nsg

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    nsg.build()
    lay, gas = W.lay, W.gas
    stream = torch.cuda.Stream()
    acc, mom, mst, g_dev, g_host = make_inputs(torch, W, stream)
    with torch.cuda.stream(stream):
        res = torch.zeros(4, dtype=torch.int32, device="cuda")
        res_host = torch.zeros(4, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    P, Q = lay.params, lay.parts
    # Up to two micro-batches: the step accumulates them itself (muon_step_ex
    # prev_grad and last_grad, the same arithmetic as muon_accumulate); they
    # overwrite accum, which the step then writes only once.  More: all of
    # them in one muon_accumulate_n pass, then the plain step -- fewer bytes
    # than folding the last two into a step that must also read and write
    # accum (four micro-batches: 12 + 8 B/elem against 8 + 16).
    nfold = gas if gas <= 2 else 0
    nacc = gas - nfold

    def fold_options(prev, last):
        if nfold == 0:
            return None
        return nsg.step_options(last_grad=last, last_grad_scale=1.0 / gas,
                                last_grad_overwrite=(gas == 1), prev_grad=prev,
                                prev_grad_scale=1.0 / gas, prev_grad_overwrite=(nacc == 0))
    fold = fold_options(g_dev[gas - 2] if nfold == 2 else None, g_dev[gas - 1])

    def step(grad_list):
        if nacc:   # all micro-batches (none folded), in one pass
            nsg.accumulate_n(acc, grad_list[:nacc], 1.0 / gas, overwrite=True, params=P, parts=Q,
                             stream=stream)
        nsg.step(acc, mom, mst, P, Q, 0.95, 0.02, W.ns_method, 5, W.clip, args.mode, result=res,
                 stream=stream, options=fold)

    # warm-up (plans are built on the first call)
    for _ in range(args.warmup):
        step(g_dev)
    torch.cuda.synchronize()
    r = nsg.read_result(res)
    if r["applied"] != 1:
        raise RuntimeError(f"warm-up step not applied: {r}")

    barrier = torch.cuda.synchronize

    # ---- the K timed steps as one CUDA graph: once the plans exist the
    # library only issues stream-ordered work (no allocation, no host
    # synchronisation), so K whole steps record into one graph and replay
    # without per-launch host overhead.  Only the Newton-Schulz launch (the
    # dominant kernel, for the roofline) is bracketed by event nodes in the
    # timed graph; the other phases are split in an eager pass afterwards.
    nsg.profile_read(reset=True)
    nsg.profile_enable(True, phases=["ns_gemm"])
    launches0 = nsg.get_stats()["kernel_launches_total"]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(args.steps):
            step(g_dev)
    launches = nsg.get_stats()["kernel_launches_total"] - launches0   # kernels of the K steps
    nsg.profile_enable(False)
    with torch.cuda.stream(stream):
        graph.replay()   # untimed: uploads the graph
    torch.cuda.synchronize()
    if nsg.read_result(res)["applied"] != 1:
        raise RuntimeError("graph replay: step not applied")
    # the event nodes are read once, after the timed replay: they then hold
    # that replay's times

    # ---- device-resident timed region: one replay = exactly K steps
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    ns_timed = nsg.profile_read(reset=True)["ns_gemm"]   # NS launches of the timed replay
    if nsg.device_error() != 0:
        raise RuntimeError("a kernel reported a device error during the timed region")
    del graph
    # phase split of the same K steps, issued eagerly with every phase's events
    nsg.profile_enable(True)
    for _ in range(args.steps):
        step(g_dev)
    torch.cuda.synchronize()
    nsg.profile_enable(False)
    phases = nsg.profile_read(reset=True)
    phases["ns_gemm"] = ns_timed

    # ---- end to end: host grads -> device, the step, result -> host.
    # Every step copies its micro-batches from pinned host memory on a copy
    # stream and reads its result back.  A micro-batch that muon_accumulate_n
    # takes is free again once accumulated, so the next step's copy into it
    # overlaps this step's Newton-Schulz; the folded ones may be read until
    # the step ends, so each alternates between two device buffers.
    # The host reads each step's result.
    h2d = sum(g.numel() * 2 for g in g_host)
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(gas)]
    consumed = [torch.cuda.Event() for _ in range(gas)]
    spare = [torch.empty_like(g_dev[i]) for i in range(nacc, gas)]
    buf = [[g_dev[i], spare[i - nacc]] if i >= nacc else [g_dev[i], g_dev[i]]
           for i in range(gas)]
    folds = [fold] + [fold_options(buf[gas - 2][1] if nfold == 2 else None, buf[gas - 1][1])]
    consumed_fold = [torch.cuda.Event() for _ in range(2)]
    res_ready = [torch.cuda.Event() for _ in range(2)]
    res_hosts = [res_host, torch.zeros(4, dtype=torch.int32).pin_memory()]
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall = time.perf_counter()
    e2.record(stream)
    copy_stream.wait_event(e2)
    copy_marks, step_marks = [], []
    for k in range(args.steps):
        b = k & 1
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(gas):
            folded = i >= nacc
            if folded and k > 1:
                copy_stream.wait_event(consumed_fold[b])
            elif not folded and k > 0:
                copy_stream.wait_event(consumed[i])
            if i == 0:
                c0.record(copy_stream)
            with torch.cuda.stream(copy_stream):
                buf[i][b if folded else 0].copy_(g_host[i], non_blocking=True)
            copied[i].record(copy_stream)
        c1.record(copy_stream)
        copy_marks.append((c0, c1))
        for mb in range(nacc):
            stream.wait_event(copied[mb])
        if nacc:
            nsg.accumulate_n(acc, g_dev[:nacc], 1.0 / gas, overwrite=True, params=P, parts=Q,
                             stream=stream)
        for mb in range(nacc):
            consumed[mb].record(stream)
        for mb in range(nacc, gas):
            stream.wait_event(copied[mb])
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        nsg.step(acc, mom, mst, P, Q, 0.95, 0.02, W.ns_method, 5, W.clip, args.mode, result=res,
                 stream=stream, options=folds[b])
        s1.record(stream)
        step_marks.append((s0, s1))
        consumed_fold[b].record(stream)
        with torch.cuda.stream(stream):
            res_hosts[k & 1].copy_(res, non_blocking=True)
        res_ready[k & 1].record(stream)
        if k > 0:
            res_ready[(k - 1) & 1].synchronize()   # the host reads the previous step's result
    e3.record(stream)
    res_ready[(args.steps - 1) & 1].synchronize()
    barrier()
    wall_ms = 1000.0 * (time.perf_counter() - t_wall) / args.steps
    e2e_ms = max(e2.elapsed_time(e3) / args.steps, wall_ms)
    if nsg.read_result(res_hosts[(args.steps - 1) & 1])["applied"] != 1:
        raise RuntimeError("end-to-end step not applied")
    # the copies' own time per step (first copy start to last copy end; a
    # copy that waits for its buffer is included from where it was issued)
    copy_list = [a.elapsed_time(b) for a, b in copy_marks]
    copy_ms = sum(copy_list) / args.steps
    step_ms_e2e = sum(a.elapsed_time(b) for a, b in step_marks) / args.steps
    # this host's plain host-to-device rate: one micro-batch copied alone,
    # after the timed loop (the first copy from a pinned buffer pays a
    # one-time cost that the steady copies do not)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(copy_stream)
    with torch.cuda.stream(copy_stream):
        buf[0][0].copy_(g_host[0], non_blocking=True)
    a1.record(copy_stream)
    a1.synchronize()
    h2d_alone_gbs = g_host[0].numel() * 2 / (a0.elapsed_time(a1) * 1e-3) / 1e9
    ws = nsg.get_stats()["workspace_bytes"]
    del acc, mom, mst, g_dev, g_host, spare, buf
    nsg.release_workspace()
    torch.cuda.empty_cache()
    return {"ms": ms, "e2e_ms": e2e_ms, "h2d": h2d, "phases": phases, "clocks": clk,
            "launches": launches, "workspace_bytes": ws, "copy_ms": copy_ms,
            "h2d_alone_gbs": h2d_alone_gbs,
            "copy_list": [round(x, 1) for x in copy_list],
            "step_ms_e2e": step_ms_e2e}


def run_dp(args, W, rank, world):
    """The data-parallel step over `world` ranks (one process per GPU, NCCL):
    the workload's parameter set cut into one partition per rank (128
    alignment), each rank holding only its own partition of accum, momentum
    and master and its partition of each micro-batch's gradients.  One step
    = the micro-batches accumulated into the local partition, then the
    data-parallel Muon step (exchange to owners, Newton-Schulz on whole
    matrices, all-reduce of the norm statistics, exchange back, write-back).
    Returns the measurements of this rank (times are maxima over ranks)."""
    import torch
    import torch.distributed as dist
    import newton_schulz_fp32_gb300 as nsg
    from newton_schulz_fp32_gb300 import dp

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    nsg.build()
    lay = wl.llama3_8b_layout(nparts=world) if W.name == "llama" else \
        wl.gpt2_small_layout(nparts=world)
    gas = W.gas
    pr = np.arange(len(lay.parts), dtype=np.int32) % world
    parts_local, sizes = dp.local_partition_table(lay.parts, pr, world)
    n = sizes[rank]
    pieces = [(int(lay.parts["storage_offset"][p]), int(parts_local["storage_offset"][p]),
               int(lay.parts["flat_end"][p] - lay.parts["flat_begin"][p]))
              for p in range(len(lay.parts)) if pr[p] == rank]
    plan = dp.DPPlan(lay.params, parts_local, pr, world, rank, W.ns_method)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        W_full = Workload(W.name, lay, gas, W.ns_method, W.clip, W.desc)
        acc_f, mom_f, mst_f, g_f, _ = make_inputs(torch, W_full, stream, host_copies=False)

        def local(t):
            out = torch.empty(n, dtype=t.dtype, device="cuda")
            for g0, l0, k in pieces:
                out[l0:l0 + k].copy_(t[g0:g0 + k])
            return out
        acc, mom, mst = local(acc_f), local(mom_f), local(mst_f)
        g_dev = [local(g) for g in g_f]
        del acc_f, mom_f, mst_f, g_f
        g_host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(gas)]
        for h, d in zip(g_host, g_dev):
            h.copy_(d)
        res = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    D = dp.DataParallelMuon(plan)

    def step():
        nsg.accumulate_n(acc, g_dev, 1.0 / gas, overwrite=True, n=n, stream=stream)
        D.step(acc, mom, mst, 0.95, 0.02, W.ns_method, 5, W.clip, args.mode, result=res,
               stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if nsg.read_result(res)["applied"] != 1:
        raise RuntimeError("warm-up step not applied")

    def barrier():
        dist.barrier()
        torch.cuda.synchronize()

    launches0 = nsg.get_stats()["kernel_launches_total"]
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    launches = nsg.get_stats()["kernel_launches_total"] - launches0
    if nsg.device_error() != 0:
        raise RuntimeError("a kernel reported a device error during the timed region")
    # end to end: the local gradients from pinned host memory every step,
    # the step, the result read back
    h2d = sum(g.numel() * 2 for g in g_host)
    res_host = torch.zeros(4, dtype=torch.int32).pin_memory()
    barrier()
    t_wall = time.perf_counter()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            for d, h in zip(g_dev, g_host):
                d.copy_(h, non_blocking=True)
        step()
        with torch.cuda.stream(stream):
            res_host.copy_(res, non_blocking=True)
        stream.synchronize()
    e3.record(stream)
    barrier()
    e2e_ms = max(e2.elapsed_time(e3) / args.steps,
                 1000.0 * (time.perf_counter() - t_wall) / args.steps)
    if nsg.read_result(res_host)["applied"] != 1:
        raise RuntimeError("end-to-end step not applied")
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], "cuda")
    return {"ms": ms, "e2e_ms": e2e_ms, "h2d": h2d, "clocks": clk, "launches": launches,
            "layout": lay, "owned_params": int(plan.sizes["owned_params"]),
            "balance": plan.sizes["owned_cost"] / max(plan.sizes["max_cost"], 1e-30),
            "exchange_elems_per_step": 2 * (plan.send_elems + plan.recv_elems)}


def host_numa():
    """The NUMA node of the GPU, the nodes of the CPUs this process may run
    on (pinned host buffers are placed near the allocating thread)."""
    out = {}
    try:
        bus = subprocess.run(["nvidia-smi", "-i", os.environ.get("LOCAL_RANK", "0"),
                              "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10).stdout.strip().lower()
        for cand in (bus, bus[4:]):
            path = f"/sys/bus/pci/devices/{cand}/numa_node"
            if cand and os.path.exists(path):
                out["gpu_node"] = int(open(path).read().strip())
                break
        cpus = os.sched_getaffinity(0)
        nodes = set()
        base = "/sys/devices/system/node"
        for nd in os.listdir(base):
            if nd.startswith("node") and nd[4:].isdigit():
                for part in open(f"{base}/{nd}/cpulist").read().strip().split(","):
                    if part:
                        a, _, b = part.partition("-")
                        if cpus & set(range(int(a), int(b or a) + 1)):
                            nodes.add(int(nd[4:]))
        out["cpu_nodes"] = sorted(nodes)
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    return out


def contract_fields(args, W, m, peaks, peak_src, world):
    """Roofline of the dominant kernel and the per-phase figures of one
    measured workload."""
    phases = m["phases"]
    lay = W.lay
    dom = max(phases, key=lambda k: phases[k]["ms"])
    ph = phases[dom]
    per_launch_ms = ph["ms"] / max(ph["launches"], 1)
    # the NS kernel runs inside seconds of back-to-back steps: the sustained
    # tensor peak is its denominator (the burst fraction is reported beside)
    if dom == "ns_gemm":
        bound, unit = "tensor", "TFLOP/s"
        achieved = (ph["flops"] / max(ph["launches"], 1)) / (per_launch_ms * 1e-3) / 1e12
        peak_key = "bf16_tflops_sustained" if W.name == "llama" else "bf16_tflops"
        peak = peak_value(peaks, peak_key) if args.mode == "bf16" else None
    else:
        bound, unit = "hbm", "GB/s"
        achieved = (ph["bytes"] / max(ph["launches"], 1)) / (per_launch_ms * 1e-3) / 1e9
        peak_key = "hbm_gbs"
        peak = peak_value(peaks, peak_key)
    roof = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_key} ({peak_src})", "unit": unit,
            "frac": (achieved / peak) if peak else None,
            "traffic": gemm_traffic(W.name) if dom == "ns_gemm" and args.mode == "bf16"
            and W.ns_method == "standard" else None,
            "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
            "work_per_launch": ph["flops"] / max(ph["launches"], 1) if dom == "ns_gemm"
            else ph["bytes"] / max(ph["launches"], 1),
            "launch_ms": per_launch_ms}
    if dom == "ns_gemm" and args.mode == "bf16" and W.ns_method == "standard" and W.name == "llama":
        ex = ns_executed_flops_pairs(lay) / (per_launch_ms * 1e-3) / 1e12
        roof["executed_tflops"] = ex   # upper tiles of the symmetric products only
        roof["executed_frac"] = ex / peak if peak else None
        roof["frac_of_burst_peak"] = achieved / peak_value(peaks, "bf16_tflops")
    hbm_phases = [k for k in phases if k != "ns_gemm" and phases[k]["ms"] > 0]
    hbm_bytes = sum(phases[k]["bytes"] for k in hbm_phases)
    hbm_ms = sum(phases[k]["ms"] for k in hbm_phases)
    ns_ms = phases["ns_gemm"]["ms"]
    ns_tflops = phases["ns_gemm"]["flops"] / max(ns_ms * 1e-3, 1e-12) / 1e12
    return {
        "ns_tflops": ns_tflops,
        "ns_frac_of_peak": (ns_tflops / peak_value(peaks, "bf16_tflops")) if args.mode == "bf16" else None,
        "ns_flops_per_step": ns_formula_flops(lay, W.ns_method),
        "hbm_gbs": hbm_bytes / max(hbm_ms * 1e-3, 1e-12) / 1e9,
        "hbm_frac_of_peak": hbm_bytes / max(hbm_ms * 1e-3, 1e-12) / 1e9 / peak_value(peaks, "hbm_gbs"),
        "phases_ms_per_step": {k: phases[k]["ms"] / args.steps for k in phases},
        "phase_gbs": {k: phases[k]["bytes"] / max(phases[k]["ms"] * 1e-3, 1e-12) / 1e9
                      for k in hbm_phases},
        "roofline": roof,
    }


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group (the
    slowest replica sets the whole job's time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def timed(torch, nsg, fn, steps, warmup, stream, prepare=None):
    """Warm-up, then CUDA-event time of `steps` calls on `stream`, with the
    library's per-phase profile over the timed calls.  prepare(), if given,
    runs before every call outside the timed spans (each call is then timed
    by its own event pair and the spans are summed)."""
    for _ in range(warmup):
        if prepare:
            prepare()
        fn()
    torch.cuda.synchronize()
    nsg.profile_read(reset=True)
    nsg.profile_enable(True)
    spans = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if prepare is None:
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
    else:
        for _ in range(steps):
            prepare()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            spans.append((a, b))
    torch.cuda.synchronize()
    nsg.profile_enable(False)
    phases = nsg.profile_read(reset=True)
    if nsg.device_error() != 0:
        raise RuntimeError("a kernel reported a device error")
    if prepare is None:
        return e0.elapsed_time(e1) / steps, phases
    return sum(a.elapsed_time(b) for a, b in spans) / steps, phases


def run_sweep(args, peaks, peak_src):
    """Newton-Schulz of single matrices (X ~ bf16 N(0,1)), one JSON line per
    shape: time per NS call and formula TFLOP/s, 5(4m^2n + 2m^3) for
    standard, 4m^2n + 34m^3 for gram."""
    import torch
    import newton_schulz_fp32_gb300 as nsg
    nsg.build()
    stream = torch.cuda.Stream()
    shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")] if args.shapes \
        else wl.SWEEP_SHAPES
    gen = torch.Generator(device="cuda").manual_seed(wl.CONFIG_SEED["sweep"])
    cpu_cache = {}
    for (r, c) in shapes:
        with torch.cuda.stream(stream):
            X = torch.randn((r, c), generator=gen, device="cuda", dtype=torch.float32)
            X = X.to(torch.bfloat16) if args.mode == "bf16" else X
            Y = torch.empty_like(X)
        torch.cuda.synchronize()
        m, n = min(r, c), max(r, c)
        flops = 5 * (4.0 * m * m * n + 2.0 * m ** 3) if args.ns_method == "standard" \
            else 4.0 * m * m * n + 34.0 * m ** 3
        ms, ph = timed(torch, nsg, lambda: nsg.newton_schulz(X, Y, args.ns_method, 5, args.mode,
                                                             stream=stream),
                       args.steps, args.warmup, stream)
        g = ph["ns_gemm"]
        tf = flops / (ms * 1e-3) / 1e12
        peak = peak_value(peaks, "bf16_tflops") if args.mode == "bf16" else None
        print(json.dumps({"metric": "NS time per matrix", "value": ms, "unit": "ms",
                          "config": {"workload": f"ns sweep {r}x{c}", "ns_method": args.ns_method,
                                     "operand_mode": args.mode},
                          "ns_tflops": tf, "frac_of_peak": (tf / peak) if peak else None,
                          "peak_source": peak_src,
                          "gemm_ms": g["ms"] / args.steps, "gemm_launches": g["launches"] / args.steps,
                          "gemm_tflops_on_gemm_time": g["flops"] / max(g["ms"] * 1e-3, 1e-12) / 1e12,
                          "cpu_baseline": None if args.no_cpu_baseline else
                          sweep_cpu_baseline(r, c, args.ns_method, args.mode, cpu_cache)}))
        del X, Y
        nsg.release_workspace()
        torch.cuda.empty_cache()


def run_ragged(args, peaks, peak_src):
    """8192 small matrices (rows {32..256} x cols {128..1024}, half tall),
    fp32 gradients written into accum, one gram Muon step."""
    import torch
    import newton_schulz_fp32_gb300 as nsg
    nsg.build()
    seed = wl.CONFIG_SEED["ragged"]
    lay = wl.ragged_layout(args.ragged_count, seed=seed)
    rng = wl.rng_for(seed, 1)
    scales = 10.0 ** rng.uniform(-5, 0, len(lay.specs))
    mats = [(wl.rng_for(seed, 2, i).standard_normal((s.rows, s.cols), dtype=np.float32)
             * np.float32(scales[i])) for i, s in enumerate(lay.specs)]
    stream = torch.cuda.Stream()
    g0 = torch.from_numpy(wl.pack(lay, mats)).cuda()
    acc = g0.clone()
    mom = torch.zeros_like(acc)
    mst = torch.zeros_like(acc)
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()

    def refill():   # the step consumes accum: fresh gradients, outside the timed span
        with torch.cuda.stream(stream):
            acc.copy_(g0)

    def step():
        nsg.step(acc, mom, mst, lay.params, lay.parts, 0.95, 0.02, "gram", 5, 0.0, args.mode,
                 result=res, stream=stream)
    ms, ph = timed(torch, nsg, step, args.steps, args.warmup, stream, prepare=refill)
    flops = ns_formula_flops(lay, "gram")
    ns_ms = ph["ns_gemm"]["ms"] / args.steps
    # the recurrence moves split-3 operands: its roofline is HBM (bytes from
    # one ncu capture of this workload, BF16 mode, 8192 matrices)
    traffic = _traffic_if_current(RAGGED_NS_TRAFFIC, "bytes_per_step") \
        if args.mode == "bf16" and args.ragged_count == 8192 else None
    hbm = peak_value(peaks, "hbm_gbs")
    print(json.dumps({"metric": "Muon step time", "value": ms, "unit": "ms",
                      "config": {"workload": f"ragged {args.ragged_count} matrices, gram NS x5",
                                 "operand_mode": args.mode,
                                 "elements": lay.n_muon_elements},
                      "ns_tflops_gram_flops": flops / (ns_ms * 1e-3) / 1e12,
                      "ns_roofline": None if traffic is None else {
                          "bound": "hbm", "achieved": traffic / (ns_ms * 1e-3) / 1e9,
                          "peak": hbm, "unit": "GB/s", "frac": traffic / (ns_ms * 1e-3) / 1e9 / hbm,
                          "traffic": traffic, "traffic_note": "DRAM bytes of the step's 16 GEMM "
                          "launches, ncu"},
                      "phases_ms_per_step": {k: ph[k]["ms"] / args.steps for k in ph},
                      "cpu_baseline": None if args.no_cpu_baseline else
                      ragged_cpu_baseline(lay, mats, args.mode, args.cpu_budget)}))


def run_llama_layers(args, peaks, peak_src):
    """A Llama-3-8B-shaped case of --layers layers (each q, o 4096^2; k, v
    1024x4096; gate, up 14336x4096; down 4096x14336; 64 partitions, align
    128; 2 bf16 micro-batches, even-indexed matrices rank 8 + 1e-3 noise),
    one standard Muon step timed eagerly.  Small enough for profiler
    captures at --layers 1; --workspace-budget runs the NS blocks in waves."""
    import torch
    import newton_schulz_fp32_gb300 as nsg
    nsg.build()
    W = llama_workload(args.mode, layers=args.layers)
    lay = W.lay
    stream = torch.cuda.Stream()
    acc, mom, mst, grads, _ = make_inputs(torch, W, stream)
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    P, Q = lay.params, lay.parts

    def step():
        nsg.step(acc, mom, mst, P, Q, 0.95, 0.02, "standard", 5, 0.0, args.mode, result=res,
                 stream=stream, options=opts)
    # both micro-batches are folded into the step;
    # --workspace-budget: the NS blocks run in waves whose workspace fits it
    opts = nsg.step_options(workspace_budget=args.workspace_budget, last_grad=grads[1],
                            last_grad_scale=0.5, prev_grad=grads[0], prev_grad_scale=0.5,
                            prev_grad_overwrite=True)
    ms, ph = timed(torch, nsg, step, args.steps, args.warmup, stream)
    flops = ns_formula_flops(lay, "standard")
    g = ph["ns_gemm"]
    hbm = [k for k in ph if k != "ns_gemm" and ph[k]["ms"] > 0]
    print(json.dumps({"metric": "Muon step time", "value": ms, "unit": "ms",
                      "config": {"workload": W.desc, "operand_mode": args.mode,
                                 "workspace_budget_bytes": args.workspace_budget},
                      "workspace_bytes": nsg.get_stats()["workspace_bytes"],
                      "ns_tflops": flops / (g["ms"] / args.steps * 1e-3) / 1e12,
                      "ns_launches_per_step": g["launches"] / args.steps,
                      "ns_flops_per_step": flops,
                      "hbm_gbs": sum(ph[k]["bytes"] for k in hbm) / (sum(ph[k]["ms"] for k in hbm) * 1e-3) / 1e9,
                      "phases_ms_per_step": {k: ph[k]["ms"] / args.steps for k in ph},
                      "result": nsg.read_result(res)}))


def reference_line(args, peaks, peak_src):
    """The reference arm: the CPU oracle on the host cores, on the workload
    this bench measures.  Each of the W + K steps is the bounded sample (the
    whole GPT-2-small step, or the first Llama-3-8B matrix of the sample
    order); the line's value is the full step extrapolated from the timed
    steps' mean; steps and ms_per_step say what was timed."""
    cores, model = cpu_info()
    if args.workload == "gpt2":
        run = lambda: (oracle_step_gpt2(args.ns_method, args.mode), 1.0, "the whole GPT-2-small step")
    else:
        total = ns_formula_flops(wl.llama3_8b_layout(), "standard")

        def run():
            sec, flops, names = oracle_step_llama_sample(args.mode, 0.0)
            return sec, total / flops, f"the whole step of one layer-0 matrix ({names[0]})"
    for _ in range(args.warmup):
        run()
    secs = []
    for _ in range(args.steps):
        sec, scale, what = run()
        secs.append(sec)
    ms_sample = 1000.0 * float(np.mean(secs))
    ms_full = ms_sample * scale
    W = gpt2_workload(args.ns_method, args.mode) if args.workload == "gpt2" else llama_workload(args.mode)
    sample = (f"oracle ({_oracle_mode(args.mode)} mode, numpy fp64 BLAS): each step times {what}; "
              f"value = mean over {args.steps} steps x {scale:.0f} (formula flops of the full "
              f"step over the sample's)")
    return {"metric": METRIC, "value": ms_full, "unit": "ms", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_sample, "sampled": scale != 1.0, "sample_scale": scale,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": args.mode + "+fp32", "data": "synthetic",
            "config": {"workload": W.desc + " (oracle on CPU, bounded sample)",
                       "ns_method": W.ns_method, "operand_mode": args.mode},
            "cpu_baseline": {"value": ms_full, "unit": "ms", "cores": cores, "cpu": model,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": ms_full, "unit": "ms", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def dp_line(args, W, m, world):
    """The contract line of a data-parallel run (N ranks, strong scaling:
    the same parameter set over more GPUs)."""
    lay = m["layout"]
    desc = W.desc.replace("P=64", f"P={world}").replace("P=8", f"P={world}")
    desc = desc.split("; the ")[0] + "; every micro-batch accumulated by muon_accumulate"
    return {
        "metric": METRIC, "value": m["ms"], "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms"], "higher_is_better": False,
        "scaling": "strong", "vs_baseline": None, "dtype": args.mode + "+fp32",
        "data": "synthetic",
        "config": {"workload": desc + "; data parallel: each rank holds one partition, "
                                      "matrices spread over owner ranks, NCCL all-to-all of "
                                      "the slices each way and one all-reduce of the norm "
                                      "statistics",
                   "parallelism": f"dp{world}", "ns_method": W.ns_method,
                   "operand_mode": args.mode,
                   "l2": f"inputs larger than L2 ({4 * lay.storage_size / world / 1e9:.2f} GB of "
                         "fp32 state per rank and buffer), no flush",
                   "launch": "eager; K steps between events, barrier on both sides, max over ranks"},
        "ns_flops_per_step": ns_formula_flops(lay, W.ns_method),
        "ns_tflops_whole_job": ns_formula_flops(lay, W.ns_method) / (m["ms"] * 1e-3) / 1e12,
        "rank0_owned_params": m["owned_params"], "rank0_load_vs_max": m["balance"],
        "exchange_elems_per_step_rank0": m["exchange_elems_per_step"],
        "roofline": None, "cpu_baseline": None,
        "e2e": {"value": m["e2e_ms"], "unit": "ms", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": 16},
        "gpu_launches": m["launches"], "clocks": m["clocks"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ns-method", default="standard", choices=["standard", "gram"],
                    help="gpt2 workload only (the Llama-3-8B config runs the standard method)")
    ap.add_argument("--mode", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle time for the Llama-3-8B cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the GPT-2-small summary inside the Llama-3-8B line")
    ap.add_argument("--workload", default="llama",
                    choices=["llama", "gpt2", "sweep", "ragged", "llama_layers"],
                    help="llama (default) and gpt2 print the contract line; sweep, ragged and "
                         "llama_layers (a smaller Llama-shaped case for profiler captures) print "
                         "extra lines")
    ap.add_argument("--layers", type=int, default=1, help="llama_layers: layers of the case")
    ap.add_argument("--dp", action="store_true",
                    help="run the data-parallel path even on one rank (one-rank NCCL group)")
    ap.add_argument("--shapes", default="", help="sweep shapes, e.g. 4096x4096,4096x16384")
    ap.add_argument("--ragged-count", type=int, default=8192,
                    help="ragged workload: number of matrices (a smaller count keeps profiler "
                         "captures small; the same shape distribution)")
    ap.add_argument("--workspace-budget", type=int, default=0,
                    help="llama_layers workload: NS workspace cap in bytes (0: unbounded)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_line(args, peaks, peak_src)))
        return
    if args.workload in ("sweep", "ragged", "llama_layers"):
        {"sweep": run_sweep, "ragged": run_ragged, "llama_layers": run_llama_layers}[
            args.workload](args, peaks, peak_src)
        return

    if world > 1 or args.dp:
        import torch
        import torch.distributed as dist
        if world == 1:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29517")
            os.environ.setdefault("RANK", "0")
            os.environ.setdefault("WORLD_SIZE", "1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))

    W = gpt2_workload(args.ns_method, args.mode) if args.workload == "gpt2" else llama_workload(args.mode)
    if world > 1 or args.dp:
        import torch.distributed as dist
        m = run_dp(args, W, rank, world)
        if rank == 0:
            print(json.dumps(dp_line(args, W, m, world)))
        dist.destroy_process_group()
        return
    m = run_gpu(args, W, rank, world)
    fields = contract_fields(args, W, m, peaks, peak_src, world)
    secondary = None
    if args.workload == "llama" and not args.no_secondary:
        G = gpt2_workload("standard", args.mode)
        mg = run_gpu(args, G, rank, world)
        fg = contract_fields(args, G, mg, peaks, peak_src, world)
        secondary = {"workload": G.desc, "ms_per_step": mg["ms"], "e2e_ms": mg["e2e_ms"],
                     "ns_tflops": fg["ns_tflops"], "ns_frac_of_peak": fg["ns_frac_of_peak"],
                     "hbm_gbs": fg["hbm_gbs"], "roofline": fg["roofline"],
                     "phases_ms_per_step": fg["phases_ms_per_step"], "clocks": mg["clocks"]}
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(W.name, W.ns_method, args.mode, args.cpu_budget)
        if secondary is not None:
            secondary["cpu_baseline"] = cpu_baseline("gpt2", "standard", args.mode, args.cpu_budget)
    line = {
        "metric": METRIC, "value": m["ms"], "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": args.mode + "+fp32",
        "data": "synthetic",
        "config": {"workload": W.desc, "parallelism": "single",
                   "l2": "inputs larger than L2 (each fp32 state buffer "
                         f"{4 * W.lay.storage_size / 1e9:.2f} GB), no flush",
                   "ns_method": W.ns_method, "operand_mode": args.mode,
                   "launch": "timed: one replay of a CUDA graph of the K steps (any accumulations + "
                             "muon_step_ex), event nodes around the NS launch only (roofline); "
                             "other phases split in an eager pass of the same K steps; e2e: "
                             "issued eagerly, with the host copies"},
        **fields,
        "workspace_bytes": m["workspace_bytes"],
        "cpu_baseline": cpu,
        "e2e": {"value": m["e2e_ms"], "unit": "ms", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": 16, "copy_stream_ms_per_step": m["copy_ms"],
                "step_call_ms_in_e2e": m["step_ms_e2e"],
                "h2d_gbs_one_copy_alone": m["h2d_alone_gbs"],
                "copy_stream_ms_each_step": m["copy_list"],
                "host_numa": host_numa()},
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
    }
    if secondary is not None:
        line["secondary"] = secondary
    print(json.dumps(line))


if __name__ == "__main__":
    main()
