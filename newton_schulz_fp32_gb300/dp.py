"""Data-parallel Muon step: the state split over ranks, one process per GPU.

Binding of the ``muon_dp_*`` calls of ``include/muon.h`` plus the order of
the collectives around them (argument marshalling and the collective calls
only; the tables come from the library's planner and every byte of the
step is moved and computed by its kernels).

Each rank holds its partitions of the flat buffers (accum, momentum,
master).  A plan assigns every parameter to one owner rank; a step then
runs, on every rank:

1. ``pack_forward``: the held slices (gradient, and momentum for Muon
   parameters) into a send buffer ordered by owner;
2. all-to-all with the plan's split sizes;
3. ``local_step``: the received slices into packed buffers of the owned
   parameters, and the library's step on them (clip 0, lr 0, statistics
   out): the unclipped update u and the new momentum m';
4. all-reduce (sum) of the four statistics: the global sum of squares, the
   skip count and the NS count;
5. ``pack_reverse``: u and m' back into the receive layout; the reverse
   all-to-all lands each slice in its holder's send layout;
6. ``finish``: the clip coefficient from the global sum, and the write-back
   of the held slices (Muon accum = coef u, master -= lr coef u,
   momentum = m'; auxiliary accum = coef g).

The phases are separate methods so that a test can run several ranks'
phases in one process and move the buffers between them itself.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import PARAM_DTYPE, PART_DTYPE, NS_METHODS, _check, _ptr, _stream, _table, lib, step_options

SEGMENT_DTYPE = np.dtype([("param", "<i4"), ("peer", "<i4"), ("is_muon", "<i4"), ("pad", "<i4"),
                          ("len", "<i8"), ("local", "<i8"), ("buf", "<i8")])
ASSIGN = {"balanced": 0, "round_robin": 1}
SEND, RECV = 0, 1


class Sizes(ctypes.Structure):
    """muon_dp_sizes_t."""
    _fields_ = [("world", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("owned_params", ctypes.c_int32), ("nparams", ctypes.c_int32),
                ("owned_elems", ctypes.c_int64), ("send_segments", ctypes.c_int64),
                ("recv_segments", ctypes.c_int64), ("send_elems", ctypes.c_int64),
                ("recv_elems", ctypes.c_int64), ("owned_cost", ctypes.c_double),
                ("max_cost", ctypes.c_double)]


_bound = False


def _bind():
    global _bound
    if _bound:
        return lib()
    L = lib()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.muon_dp_plan_create.argtypes = [P, I, P, P, I, I, I, I, I, ctypes.POINTER(P)]
    L.muon_dp_plan_destroy.argtypes = [P]
    L.muon_dp_plan_destroy.restype = None
    L.muon_dp_plan_sizes.argtypes = [P, ctypes.POINTER(Sizes)]
    L.muon_dp_plan_tables.argtypes = [P, P, P, P, P, P, P]
    L.muon_dp_pack.argtypes = [P, I, P, P, P, P]
    L.muon_dp_unpack.argtypes = [P, I, P, P, P, P]
    L.muon_dp_finish.argtypes = [P, P, P, P, P, P, F, F, P, P]
    for name in ("muon_dp_plan_create", "muon_dp_plan_sizes", "muon_dp_plan_tables",
                 "muon_dp_pack", "muon_dp_unpack", "muon_dp_finish"):
        getattr(L, name).restype = I
    _bound = True
    return L


class DPPlan:
    """The plan of one rank (host tables; no GPU needed to build it).

    params, parts: the whole model's tables (PARAM_DTYPE, PART_DTYPE), with
    each partition's storage_offset an index into its holder's buffers;
    part_rank[p]: the rank holding partition p."""

    def __init__(self, params, parts, part_rank, world: int, rank: int, ns_method="gram",
                 assign="balanced"):
        L = _bind()
        p, self.nparams = _table(params, PARAM_DTYPE)
        q, nq = _table(parts, PART_DTYPE)
        pr = np.ascontiguousarray(part_rank, dtype=np.int32)
        if len(pr) != nq:
            raise ValueError("part_rank needs one entry per partition")
        method = NS_METHODS[ns_method] if isinstance(ns_method, str) else int(ns_method)
        h = ctypes.c_void_p()
        _check(L.muon_dp_plan_create(p.ctypes.data if self.nparams else None, self.nparams,
                                     q.ctypes.data if nq else None,
                                     pr.ctypes.data if nq else None, nq, world, rank, method,
                                     ASSIGN[assign], ctypes.byref(h)))
        self.handle = h
        s = Sizes()
        _check(L.muon_dp_plan_sizes(h, ctypes.byref(s)))
        self.sizes = {k: getattr(s, k) for k, _ in Sizes._fields_}
        self.world, self.rank = world, rank
        self.owner = np.zeros(self.nparams, np.int32)
        self.send_counts = np.zeros(world, np.int64)
        self.recv_counts = np.zeros(world, np.int64)
        self.owned_params = np.zeros(s.owned_params, PARAM_DTYPE)
        self.send_segs = np.zeros(s.send_segments, SEGMENT_DTYPE)
        self.recv_segs = np.zeros(s.recv_segments, SEGMENT_DTYPE)
        arr = lambda a: a.ctypes.data if a.size else None
        _check(L.muon_dp_plan_tables(h, arr(self.owner), arr(self.send_counts),
                                     arr(self.recv_counts), arr(self.owned_params),
                                     arr(self.send_segs), arr(self.recv_segs)))
        self.owned_elems = int(s.owned_elems)
        self.send_elems, self.recv_elems = int(s.send_elems), int(s.recv_elems)
        # the packed owned buffers: one partition [0, owned_elems), storage 0
        self.owned_parts = np.zeros(1 if self.owned_elems else 0, PART_DTYPE)
        if self.owned_elems:
            self.owned_parts[0] = (0, self.owned_elems, 0)

    def close(self):
        if self.handle:
            _bind().muon_dp_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DataParallelMuon:
    """The data-parallel step of one rank on CUDA tensors.

    accum, momentum, master: this rank's storage buffers (float32, 16-byte
    aligned).  Buffers for the exchanges and the owned parameters are
    allocated once, here (torch's allocator)."""

    def __init__(self, plan: DPPlan, device=None, workspace_budget: int = 0):
        import torch
        self.plan = plan
        self.torch = torch
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        f32 = dict(dtype=torch.float32, device=dev)
        n4 = lambda n: max(4, (n + 3) // 4 * 4)
        self.send = torch.zeros(n4(plan.send_elems), **f32)
        self.recv = torch.zeros(n4(plan.recv_elems), **f32)
        self.own_acc = torch.zeros(n4(plan.owned_elems), **f32)
        self.own_mom = torch.zeros(n4(plan.owned_elems), **f32)
        self.own_mst = torch.zeros(n4(plan.owned_elems), **f32)
        self.stats = torch.zeros(4, dtype=torch.float64, device=dev)
        self.local_result = torch.zeros(4, dtype=torch.int32, device=dev)
        self.workspace_budget = int(workspace_budget)

    # ---- phases
    def pack_forward(self, accum, momentum, stream=None):
        _check(_bind().muon_dp_pack(self.plan.handle, SEND, _ptr(self.send), _ptr(accum),
                                    _ptr(momentum), _stream(stream)))
        return self.send

    def local_step(self, beta, ns_method="gram", ns_steps=5, operand_mode="bf16",
                   grad_scale=1.0, stream=None):
        """Receive buffer -> owned buffers, then the library's step on the
        owned parameters with clip 0 and lr 0; fills self.stats."""
        L = _bind()
        _check(L.muon_dp_unpack(self.plan.handle, RECV, _ptr(self.recv), _ptr(self.own_acc),
                                _ptr(self.own_mom), _stream(stream)))
        opts = step_options(grad_scale=grad_scale, workspace_budget=self.workspace_budget,
                            stats_out=self.stats)
        from . import step
        step(self.own_acc, self.own_mom, self.own_mst, self.plan.owned_params,
             self.plan.owned_parts, beta, 0.0, ns_method, ns_steps, 0.0, operand_mode,
             result=self.local_result, stream=stream, options=opts)
        return self.stats

    def pack_reverse(self, stream=None):
        _check(_bind().muon_dp_pack(self.plan.handle, RECV, _ptr(self.recv), _ptr(self.own_acc),
                                    _ptr(self.own_mom), _stream(stream)))
        return self.recv

    def finish(self, accum, momentum, master, lr, clip, result, stream=None):
        _check(_bind().muon_dp_finish(self.plan.handle, _ptr(self.send), _ptr(accum),
                                      _ptr(momentum), _ptr(master), _ptr(self.stats), lr, clip,
                                      _ptr(result), _stream(stream)))
        return result

    # ---- the step with torch.distributed collectives
    def step(self, accum, momentum, master, beta, lr, ns_method="gram", ns_steps=5, clip=0.0,
             operand_mode="bf16", grad_scale=1.0, result=None, group=None, stream=None):
        """One data-parallel Muon step (all ranks of `group` call it)."""
        torch = self.torch
        if result is None:
            result = torch.zeros(4, dtype=torch.int32, device=accum.device)
        s = stream if stream is not None else torch.cuda.current_stream()
        dp = self

        class Phases:
            send = dp.send[:dp.plan.send_elems]
            recv = dp.recv[:dp.plan.recv_elems]
            stats = dp.stats

            def pack_forward(self):
                dp.pack_forward(accum, momentum, s)

            def local_step(self):
                dp.local_step(beta, ns_method, ns_steps, operand_mode, grad_scale, s)

            def pack_reverse(self):
                dp.pack_reverse(s)

            def finish(self):
                dp.finish(accum, momentum, master, lr, clip, result, s)

        with torch.cuda.stream(s):
            exchange(Phases(), self.plan, group)
        return result


def exchange(phases, plan, group=None):
    """The collective order of one data-parallel step around one rank's
    phases: pack, all-to-all (split sizes from the plan), the owners' local
    step, all-reduce (sum) of the statistics, pack of the results,
    all-to-all back (split sizes swapped), write-back.  `phases` has the
    exchange tensors send, recv and stats and the four phase methods."""
    import torch.distributed as dist
    sc, rc = plan.send_counts.tolist(), plan.recv_counts.tolist()
    phases.pack_forward()
    dist.all_to_all_single(phases.recv, phases.send, rc, sc, group=group)
    phases.local_step()
    dist.all_reduce(phases.stats, op=dist.ReduceOp.SUM, group=group)
    phases.pack_reverse()
    dist.all_to_all_single(phases.send, phases.recv, sc, rc, group=group)
    phases.finish()


def local_partition_table(layout_parts, part_rank, world: int):
    """The partition table every rank's plan takes: each partition's
    storage_offset is its place in its holder's buffers (partitions of one
    rank back to back in flat order).  Returns (parts, storage size per
    rank)."""
    parts = np.array(layout_parts, dtype=PART_DTYPE, copy=True)
    sizes = [0] * world
    for p in range(len(parts)):
        r = int(part_rank[p])
        parts["storage_offset"][p] = sizes[r]
        sizes[r] += int(parts["flat_end"][p] - parts["flat_begin"][p])
    return parts, sizes
