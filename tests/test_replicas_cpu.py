"""The bench's multi-GPU line takes the slowest rank's time for the whole
job (the maximum of the per-rank times over the process group).  Checked
here with two gloo processes on the CPU; the data-parallel step's own
exchange is tested in test_dp_cpu.py."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks([1.5 + rank, 10.0 - rank, 3.25], "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # every rank gets the slowest replica's value for each entry
    assert res[0] == res[1] == [2.5, 10.0, 3.25]
