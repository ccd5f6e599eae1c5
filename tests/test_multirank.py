"""The N > 1 bench path on the CPU: two gloo ranks, each with its own layer
(replicas, no collective on the data path).  The job time is the slowest
rank's, and the reported value is seconds per layer over all ranks' layers."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [120.0, 95.0][rank]  # the first rank is slower
    job_ms = bench.max_over_ranks(local_ms, world)
    out[rank] = (job_ms, bench.seconds_per_layer(job_ms / 10, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        job_ms, spl = res[rank]
        assert job_ms == 120.0
        assert spl == pytest.approx(120.0 / 10 / 1e3 / 2)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(42.0, 1) == 42.0
    assert bench.seconds_per_layer(8.0, 1) == pytest.approx(0.008)
