"""The multi-process path of bench.py on the CPU: two gloo ranks (replicas)
agree on the slowest replica's time, pass the barrier, and only rank 0 of
the reference arm does any work."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    import bench
    bench.barrier_ranks(world)
    # each rank's step time; every rank must see the slowest one
    t_max = bench.max_over_ranks(1.5 * (rank + 1), world, torch.device("cpu"))
    # the reference arm runs on rank 0 only; other ranks return at once
    ref_rc = None
    if rank != 0:
        args = type("A", (), dict(workload="tiny", steps=1, warmup=0,
                                  gpus=world))()
        ref_rc = bench.run_reference(args)
    bench.barrier_ranks(world)
    dist.destroy_process_group()
    out.put((rank, t_max, ref_rc))


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out))
             for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, t_max, ref_rc = out.get(timeout=120)
        res[rank] = (t_max, ref_rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == pytest.approx(3.0) and res[1][0] == pytest.approx(3.0)
    assert res[1][1] == 0


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier_ranks(1)
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
