"""The multi-rank bench path on CPU: two gloo ranks agree on the slowest rank's step time and on
the whole-job throughput (weak scaling: every rank moves the same per-GPU bytes; no collective
touches the data path, only this timing reduction)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    ms = bench.max_over_ranks(1.0 + 2.0 * rank, world)  # rank 1 is the slow one
    out[rank] = (ms, bench.weak_scaling_value(10 ** 9, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    ms, gbs = res[0]
    assert ms == 3.0
    assert abs(gbs - 2 * 1e9 / 3e-3 / 1e9) < 1e-9


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.weak_scaling_value(10 ** 9, 1.0, 1) == 1000.0
