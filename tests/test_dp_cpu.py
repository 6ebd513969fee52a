"""Data parallelism across ranks, on the CPU: the library's planner (host
only, no CUDA call) and the exchange order of newton_schulz_fp32_gb300.dp
run by two and three gloo processes.

The planner's tables are checked for consistency between ranks (what s
sends to d is what d expects from s, slice by slice), for exact coverage of
every parameter at its owner, and for the assignment's balance.  The
exchange is then run for real with torch.distributed (gloo): each rank
keeps only its own partitions of the tiny and GPT-2-layer configurations,
packs its slices by the plan, the owners run the oracle's Muon update on
the whole matrices they receive, per-parameter sums of squares are
all-reduced (each entry has exactly one non-zero contributor, so the sum
is exact) and added up in table order, and the write-back lands in every
rank's partitions.  The result must equal the single-process oracle step
on the whole flat buffer bit for bit -- the pages' multi-GPU check ("Support
Muon in BF16_Optimizer with FP32 gradient accumulation", validation table:
weights and momentum against the reference, max error 0.0)."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import newton_schulz_fp32_gb300 as nsg  # noqa: E402
from newton_schulz_fp32_gb300 import dp  # noqa: E402
from oracle import muon as om  # noqa: E402
import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def library():
    nsg.build()


def part_ranks(lay):
    """Partition p of each segment is held by rank p (the layouts cut every
    segment into nparts equal partitions, one per rank)."""
    return np.arange(len(lay.parts), dtype=np.int32) % lay.nparts


LAYOUTS = {
    "tiny": lambda w: wl.tiny_layout(nparts=w),
    "gpt2_layer": lambda w: wl.gpt2_small_layout(layers=1, nparts=w),
    "ragged64": lambda w: wl.ragged_layout(64, nparts=w),
    "llama_layer": lambda w: wl.llama3_8b_layout(layers=1, nparts=w),
}


def up4(n):
    return (n + 3) // 4 * 4


# ------------------------------------------------------------ the planner

@pytest.mark.parametrize("name", list(LAYOUTS))
@pytest.mark.parametrize("world", [1, 2, 3, 5])
@pytest.mark.parametrize("assign", ["balanced", "round_robin"])
def test_plan_tables_agree_between_ranks(name, world, assign):
    lay = LAYOUTS[name](world)
    pr = part_ranks(lay)
    parts, sizes = dp.local_partition_table(lay.parts, pr, world)
    plans = [dp.DPPlan(lay.params, parts, pr, world, r, "gram", assign) for r in range(world)]
    n = len(lay.params)
    numel = lay.params["rows"].astype(np.int64) * lay.params["cols"]
    for p in plans[1:]:
        assert np.array_equal(p.owner, plans[0].owner)
    owner = plans[0].owner
    assert owner.min() >= 0 and owner.max() < world
    if assign == "round_robin":
        assert np.array_equal(owner, np.arange(n) % world)
    for s in range(world):
        for d in range(world):
            assert plans[s].send_counts[d] == plans[d].recv_counts[s]
            snd = plans[s].send_segs[plans[s].send_segs["peer"] == d]
            rcv = plans[d].recv_segs[plans[d].recv_segs["peer"] == s]
            # the same slices in the same order on both sides
            assert np.array_equal(snd["param"], rcv["param"])
            assert np.array_equal(snd["len"], rcv["len"])
            assert np.array_equal(snd["is_muon"], rcv["is_muon"])
    for r, p in enumerate(plans):
        for segs, total in ((p.send_segs, p.send_elems), (p.recv_segs, p.recv_elems)):
            # buffers: 4-aligned slices back to back, peers in rank order
            off = 0
            for sg in segs:
                assert sg["buf"] == off and sg["buf"] % 4 == 0
                off += up4(int(sg["len"])) * (2 if sg["is_muon"] else 1)
            assert off == total
            assert np.all(np.diff(segs["peer"]) >= 0)
        assert np.all(p.send_segs["local"] + p.send_segs["len"] <= sizes[r])
        assert np.all(p.send_segs["is_muon"] == lay.params["use_muon"][p.send_segs["param"]])
        # owned parameters: table order, 32-element aligned, each covered
        # exactly once by the received slices
        mine = np.flatnonzero(owner == r)
        assert len(p.owned_params) == len(mine)
        assert np.all(p.owned_params["offset"] % 32 == 0)
        cover = np.zeros(p.owned_elems, np.int32)
        for sg in p.recv_segs:
            cover[sg["local"]:sg["local"] + sg["len"]] += 1
        for q, k in zip(p.owned_params, mine):
            assert (q["rows"], q["cols"]) == (lay.params["rows"][k], lay.params["cols"][k])
            assert np.all(cover[q["offset"]:q["offset"] + numel[k]] == 1)
        assert cover.sum() == numel[mine].sum()
        p.close()


@pytest.mark.parametrize("name", ["gpt2_layer", "llama_layer", "ragged64"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_balanced_assignment_within_the_lpt_bound(name, world):
    """Largest first onto the least loaded rank is within the largest item
    of the perfect split (Graham's bound for this greedy order)."""
    lay = LAYOUTS[name](world)
    pr = part_ranks(lay)
    parts, _ = dp.local_partition_table(lay.parts, pr, world)
    p = dp.DPPlan(lay.params, parts, pr, world, 0, "standard", "balanced")
    rr = dp.DPPlan(lay.params, parts, pr, world, 0, "standard", "round_robin")
    costs = []
    for k in range(len(lay.params)):
        rows, cols, h = (int(lay.params[f][k]) for f in ("rows", "cols", "num_heads"))
        h = max(h, 1) if lay.params["use_muon"][k] else 1
        r, c = rows // h, cols
        m, n = min(r, c), max(r, c)
        f = h * 5 * (4.0 * m * m * n + 2.0 * m ** 3) if lay.params["use_muon"][k] else 0.0
        costs.append(f + 12500.0 * rows * cols)
    total, big = sum(costs), max(costs)
    assert p.sizes["max_cost"] <= total / world + big + 1e-6 * total
    assert p.sizes["max_cost"] <= rr.sizes["max_cost"] * (1 + 1e-12)
    p.close()
    rr.close()


def test_plan_rejects_bad_tables():
    lay = wl.tiny_layout(nparts=2)
    pr = part_ranks(lay)
    parts, _ = dp.local_partition_table(lay.parts, pr, 2)
    bad = pr.copy()
    bad[0] = 2
    with pytest.raises(nsg.MuonError, match="part_rank"):
        dp.DPPlan(lay.params, parts, bad, 2, 0)
    clash = parts.copy()
    clash["storage_offset"][2] = 0          # rank 0's second partition over its first
    with pytest.raises(nsg.MuonError, match="overlap in storage"):
        dp.DPPlan(lay.params, clash, pr, 2, 0)
    with pytest.raises(nsg.MuonError, match="not covered"):
        dp.DPPlan(lay.params, parts[1:], pr[1:], 2, 0)
    with pytest.raises(nsg.MuonError, match="rank"):
        dp.DPPlan(lay.params, parts, pr, 2, 2)


# ------------------------------------------------------------ the exchange, with gloo

class OraclePhases:
    """One rank's phases on the CPU: copies by the plan's segments, the
    oracle's update at the owners, statistics per parameter (float64
    buffers, so an exact-mode update crosses the exchange unrounded)."""

    def __init__(self, plan, lay, acc, mom, mst, beta, lr, method, mode, clip):
        self.plan, self.lay = plan, lay
        self.acc, self.mom, self.mst = acc, mom, mst
        self.beta, self.lr, self.method, self.mode, self.clip = beta, lr, method, mode, clip
        self.n = len(lay.params)
        self.send = torch.zeros(plan.send_elems, dtype=torch.float64)
        self.recv = torch.zeros(plan.recv_elems, dtype=torch.float64)
        self.stats = torch.zeros(self.n + 1, dtype=torch.float64)   # per-parameter sums, skips
        self.mine = np.flatnonzero(plan.owner == plan.rank)

    def pack_forward(self):
        s = self.send.numpy()
        for sg in self.plan.send_segs:
            b, L, loc = int(sg["buf"]), int(sg["len"]), int(sg["local"])
            s[b:b + L] = self.acc[loc:loc + L]
            if sg["is_muon"]:
                s[b + up4(L):b + up4(L) + L] = self.mom[loc:loc + L]

    def local_step(self):
        r = self.recv.numpy()
        own_g = np.zeros(self.plan.owned_elems)
        own_m = np.zeros(self.plan.owned_elems)
        for sg in self.plan.recv_segs:
            b, L, loc = int(sg["buf"]), int(sg["len"]), int(sg["local"])
            own_g[loc:loc + L] = r[b:b + L]
            if sg["is_muon"]:
                own_m[loc:loc + L] = r[b + up4(L):b + up4(L) + L]
        st = self.stats.numpy()
        st[:] = 0.0
        for q, k in zip(self.plan.owned_params, self.mine):
            o, rows, cols = int(q["offset"]), int(q["rows"]), int(q["cols"])
            g = own_g[o:o + rows * cols].astype(np.float32).reshape(rows, cols)
            if not np.all(np.isfinite(g)):
                st[self.n] += 1.0
                continue
            if q["use_muon"]:
                m = own_m[o:o + rows * cols].astype(np.float32).reshape(rows, cols)
                m_new, u = om.muon_update(g, m, self.beta, self.method, 5, int(q["num_heads"]),
                                          self.mode)
                own_m[o:o + rows * cols] = m_new.reshape(-1)
            else:
                u = g
            u64 = np.asarray(u, np.float64)
            st[k] = float(np.sum(u64 * u64))
            own_g[o:o + rows * cols] = u64.reshape(-1)
        self.own_g, self.own_m = own_g, own_m

    def pack_reverse(self):
        r = self.recv.numpy()
        for sg in self.plan.recv_segs:
            b, L, loc = int(sg["buf"]), int(sg["len"]), int(sg["local"])
            r[b:b + L] = self.own_g[loc:loc + L]
            if sg["is_muon"]:
                r[b + up4(L):b + up4(L) + L] = self.own_m[loc:loc + L]

    def finish(self):
        st = self.stats.numpy()
        if st[self.n] > 0:
            return
        sq = 0.0
        for k in range(self.n):          # table order, as the oracle adds them
            sq += float(st[k])
        norm = float(np.sqrt(sq))
        coef = min(1.0, self.clip / (norm + om.CLIP_EPS)) if self.clip > 0 else 1.0
        s = self.send.numpy()
        for sg in self.plan.send_segs:
            b, L, loc = int(sg["buf"]), int(sg["len"]), int(sg["local"])
            u = s[b:b + L] if self.mode == "exact" else s[b:b + L].astype(np.float32)
            v, w = om.write_back(u, self.mst[loc:loc + L], coef, self.lr, self.mode,
                                 bool(sg["is_muon"]))
            self.acc[loc:loc + L] = v
            if sg["is_muon"]:
                self.mst[loc:loc + L] = w
                self.mom[loc:loc + L] = s[b + up4(L):b + up4(L) + L].astype(np.float32)


def local_view(lay, parts_local, pr, rank, glob, size):
    """A rank's own storage buffer, cut from a whole-model storage buffer."""
    out = np.zeros(size, np.float32)
    for p in range(len(lay.parts)):
        if pr[p] == rank:
            n = int(lay.parts["flat_end"][p] - lay.parts["flat_begin"][p])
            g0, l0 = int(lay.parts["storage_offset"][p]), int(parts_local["storage_offset"][p])
            out[l0:l0 + n] = glob[g0:g0 + n]
    return out


CASES = [
    # layout, method, mode, steps, clip, nan_at_step
    ("tiny", "gram", "bf16", 3, 0.05, None),
    ("tiny", "standard", "exact", 3, 0.05, None),
    ("tiny", "gram", "exact", 2, 0.0, None),
    ("tiny", "standard", "bf16", 3, 0.05, 1),
    ("gpt2_layer", "standard", "bf16", 1, 0.05, None),
]


def _dp_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        results = []
        for ci, (name, method, mode, steps, clip, nan_step) in enumerate(CASES):
            lay = LAYOUTS[name](world)
            pr = part_ranks(lay)
            parts_local, sizes = dp.local_partition_table(lay.parts, pr, world)
            plan = dp.DPPlan(lay.params, parts_local, pr, world, rank, method)
            seed = 4000 + ci
            z = [np.zeros((s.rows, s.cols), np.float32) for s in lay.specs]
            w0 = [(0.02 * wl.rng_for(seed, 9, i).standard_normal((s.rows, s.cols))).astype(np.float32)
                  for i, s in enumerate(lay.specs)]
            g_mom = wl.storage_with_sentinels(lay, z)
            g_mst = wl.storage_with_sentinels(lay, w0)
            mom = local_view(lay, parts_local, pr, rank, g_mom, sizes[rank])
            mst = local_view(lay, parts_local, pr, rank, g_mst, sizes[rank])
            ok = True
            for st in range(steps):
                grads = wl.gaussian_grads(lay, seed, st)
                if nan_step == st:
                    grads[0][1, 2] = np.nan
                g_acc = wl.storage_with_sentinels(lay, grads)
                acc = local_view(lay, parts_local, pr, rank, g_acc, sizes[rank])
                ref = om.muon_step_flat(g_acc, g_mom, g_mst, lay.params, lay.parts, 0.95, 0.02,
                                        method, 5, clip, mode)
                dp.exchange(OraclePhases(plan, lay, acc, mom, mst, 0.95, 0.02, method, mode, clip),
                            plan)
                for mine, glob in ((acc, ref[0]), (mom, ref[1]), (mst, ref[2])):
                    want = local_view(lay, parts_local, pr, rank, glob, sizes[rank])
                    ok = ok and np.array_equal(mine.view(np.uint32), want.view(np.uint32))
                ok = ok and ref[3]["applied"] == (0 if nan_step == st else 1)
                g_mom, g_mst = ref[1], ref[2]
            results.append(ok)
            plan.close()
        out[rank] = results
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_exchange_matches_single_process_oracle_bitwise(world):
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_dp_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == [True] * len(CASES), (r, res[r])


def test_plan_of_degenerate_tables():
    """An empty table, and a table of auxiliary parameters only: every rank's
    plan is consistent and owns what it should."""
    empty = wl.build_layout([[]], 128, 2)
    pr = part_ranks(empty) if len(empty.parts) else np.zeros(0, np.int32)
    parts, _ = dp.local_partition_table(empty.parts, pr, 2)
    for r in range(2):
        p = dp.DPPlan(empty.params, parts, pr, 2, r)
        assert p.owned_elems == 0 and p.send_elems == 0 and p.recv_elems == 0
        p.close()
    aux = wl.build_layout([[wl.ParamSpec("ln", 1, 768, use_muon=False),
                            wl.ParamSpec("emb", 40, 96, use_muon=False)]], 128, 3)
    pr = part_ranks(aux)
    parts, _ = dp.local_partition_table(aux.parts, pr, 3)
    plans = [dp.DPPlan(aux.params, parts, pr, 3, r) for r in range(3)]
    assert sum(p.sizes["owned_params"] for p in plans) == 2
    for p in plans:
        assert not p.send_segs["is_muon"].any() and not p.recv_segs["is_muon"].any()
        p.close()
