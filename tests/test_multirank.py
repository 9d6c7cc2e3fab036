"""The multi-process host path of bench.py on CPU (gloo, world size 2).

Every rank runs its own replica of the workload; the only exchanges are the
timing barrier and the maximum of the per-rank times, and the whole-job rate
counts the work of all ranks.  These tests start two ranks as local processes
on 127.0.0.1 and check those host-side pieces without a GPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, local, d = bench.dist_setup()
    assert d is not None and (r, w) == (rank, world)
    per_rank_ms = [3.0, 5.0][rank]
    bench.barrier(d)
    m = bench.reduce_max(per_rank_ms, d, torch.device("cpu"))
    flops_per_rank = 1e9
    value = w * flops_per_rank / (m * 1e-3) / 1e12  # whole-job TFLOP/s, as bench.py computes it
    q.put((rank, m, value))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, value in res:
        assert m == 5.0                      # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1e9 / 5e-3 / 1e12)  # both replicas' work over the slowest rank


def test_single_process_defaults():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    import bench

    r, w, local, d = bench.dist_setup()
    assert (r, w, local, d) == (0, 1, 0, None)
    assert bench.reduce_max(2.5, None, torch.device("cpu")) == 2.5
