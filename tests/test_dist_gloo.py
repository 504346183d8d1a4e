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


class _StubMap:
    def __init__(self, base, nbox, box_bytes):
        self.base, self.num_boxes, self.box_bytes, self.path = base, nbox, box_bytes, 1


class _StubTm:
    """The library's encode call, recorded on the host: each map remembers the buffer address it
    was given (what the real tmap_encode writes into the descriptor)."""
    TM_BF16, TM_F32, TM_S32 = 9, 7, 3
    TM_OOB_ZERO, TM_OOB_NAN = 0, 1
    TM_SWIZZLE_128B = 3
    ESIZE = {9: 2, 7: 4, 3: 4}

    def tmap_encode(self, dtype, buf, dims, strides, box, element_strides=None, swizzle=0, oob=0):
        nbox, bb = 1, self.ESIZE[dtype]
        for d, b in zip(dims, box):
            nbox *= -(-d // b)
            bb *= b
        return _StubMap(buf.data_ptr(), nbox, bb)


def _binding_rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bound = []
    torch.cuda.set_device = bound.append  # the device layer, stubbed: record what is selected
    _, w, local = bench.dist_env()
    device = bench.bind_device(w, local)
    # bench.py's setup path over this rank's buffers (on the CPU here, with the encoder stubbed)
    h = bench.HostWorkload(scale=64)
    g = bench.GpuWorkload(h, None, device=torch.device("cpu"), tm=_StubTm())
    g.check_rank_local()  # every map describes one of this rank's own buffers
    caught = []
    foreign = torch.zeros(64, dtype=torch.uint8)  # not one of the workload's buffers
    g.maps["peer"] = _StubTm().tmap_encode(_StubTm.TM_BF16, foreign, [32], [], [32])
    try:
        g.check_rank_local()
    except RuntimeError as e:
        caught.append(str(e))
    del g.maps["peer"]
    g.t["elsewhere"] = torch.empty(16, device="meta")  # a buffer on another device
    try:
        g.check_rank_local()
    except RuntimeError as e:
        caught.append(str(e))
    everyone = [None] * world
    dist.all_gather_object(everyone, (bound, str(device)))
    out[rank] = (everyone, caught, len(g.maps))
    dist.barrier()
    dist.destroy_process_group()


def test_each_gloo_rank_binds_its_own_device_and_buffers():
    """Two gloo ranks run the bench's device binding and workload setup (device layer and encoder
    stubbed on the CPU): rank r selects cuda:r and nothing else, every map of a rank describes one
    of that rank's own buffers, and the setup check refuses a map over a buffer the rank does not
    own or a buffer on another device.  The path is replicas: no rank's kernel ever gets a peer's
    memory."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_binding_rank, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    for rank in range(2):
        everyone, caught, nmaps = res[rank]
        assert everyone == [([0], "cuda:0"), ([1], "cuda:1")]
        assert nmaps > 10
        assert len(caught) == 2
        assert "does not describe a buffer of this rank" in caught[0]
        assert "not on this rank's" in caught[1]
