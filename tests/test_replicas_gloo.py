"""The multi-GPU path of bench.py is replicas only: every rank serves its own
requests, and the process group carries nothing but the timing barrier and
the max over ranks.  Checked here with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, local = bench.rank_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    wids = bench.replica_wids(r, 8)
    gathered = [None] * w
    dist.all_gather_object(gathered, wids)
    slowest = bench.max_over_ranks(1.0 + r, w)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, local, gathered, slowest))


def test_two_gloo_ranks_shard_requests_and_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, local, gathered, slowest in res:
        assert local == r
        assert slowest == 2.0
        assert gathered[0] == list(range(8)) and gathered[1] == list(range(8, 16))


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) is None  # returns before touching the workload
