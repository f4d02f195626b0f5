"""Host side of the multi-replica benchmark (one independent replica per
rank, no collective on the data path): two gloo ranks on the CPU agree on
the slowest replica's step time, and the rank/world environment is read the
way torchrun sets it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from conftest import ROOT  # noqa: E402
import sys  # noqa: E402

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        ms = 1.5 + 2.0 * r            # rank 1 is the slow replica
        out[r] = bench.max_over_ranks(torch, ms, w, "cpu")
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_replica_needs_no_collective():
    assert bench.max_over_ranks(torch, 2.25, 1, "cpu") == 2.25
