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


# ------------------------------------------- one layer split over ranks (CPU, gloo)
def test_token_and_row_ranges_cover_everything_once():
    sys.path.insert(0, ROOT)
    from post_weight_quantization_30_b300 import sharding as sh

    for n in (0, 1, 31, 1000, 8192, 262144, 262145):
        for world in (1, 2, 3, 4, 7, 8):
            for mult in (1, 64, 8192):
                seen = []
                for r in range(world):
                    t0, t1 = sh.token_range(n, world, r, mult)
                    assert t0 <= t1 and (t0 % mult == 0 or t0 == n)
                    seen.extend(range(t0, t1))
                assert seen == list(range(n))
    for rows in (32, 4096, 11008, 29568):
        for world in (1, 2, 3, 8):
            rr = [sh.row_range(rows, world, r) for r in range(world)]
            assert rr[0][0] == 0 and rr[-1][1] == rows
            assert all(a[1] == b[0] for a, b in zip(rr, rr[1:]))
            assert all(r0 % 32 == 0 and (r1 - r0) % 32 == 0 for r0, r1 in rr)
    with pytest.raises(ValueError):
        sh.row_range(100, 2, 0)


def _oracle_accumulate(H, X):
    from oracle import gptq as og

    H += torch.from_numpy(og.hessian(X.numpy()))


def _oracle_quantize(W, H, bits, group, block, damp):
    from oracle import gptq as og
    from oracle import pack as opk

    q = og.quantize_layer(W.numpy(), H.numpy(), bits, group, damp)
    return dict(qweight=torch.from_numpy(opk.pack_qweight(q["codes"], bits)), scales=torch.from_numpy(q["scales"]),
                qzeros=torch.from_numpy(opk.pack_qzeros(q["zeros"], bits)), codes=torch.from_numpy(q["codes"]))


SPLIT = dict(rows=96, cols=128, n=3000, bits=3, group=64)


def _split_inputs():
    import numpy as np

    rng = np.random.default_rng(5)
    X = rng.integers(-3, 4, (SPLIT["n"], SPLIT["cols"])).astype(np.float64)  # integer-valued: every sum exact
    X[:, 7] *= 9.0
    W = rng.standard_normal((SPLIT["rows"], SPLIT["cols"])) * 0.02
    return torch.from_numpy(X), torch.from_numpy(W)


def _split_rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from post_weight_quantization_30_b300 import sharding as sh

    X, W = _split_inputs()
    t0, t1 = sh.token_range(X.shape[0], world, rank, multiple=64)
    H = sh.hessian_sharded(X[t0:t1], SPLIT["cols"], accumulate=_oracle_accumulate)
    (r0, r1), q = sh.quantize_rows(W, H, SPLIT["bits"], SPLIT["group"], quantize=_oracle_quantize)
    full = sh.gather_rows(q, SPLIT["rows"], SPLIT["bits"])
    out[rank] = (t0, t1, r0, r1, H.numpy(), {k: v.numpy() for k, v in full.items()})
    dist.barrier()
    dist.destroy_process_group()


def test_split_layer_equals_single_rank_result():
    """Two gloo ranks: the token shards' H summed by the all-reduce equals the single-rank H bit for
    bit (integer-valued X), and the row shards quantized against it and gathered equal the single-rank
    quantization bit for bit (rows are independent given H).  The per-shard work is the oracle's."""
    import numpy as np

    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_split_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    sys.path.insert(0, ROOT)
    X, W = _split_inputs()
    H1 = torch.zeros((SPLIT["cols"], SPLIT["cols"]), dtype=torch.float64)
    _oracle_accumulate(H1, X)
    ref = _oracle_quantize(W, H1, SPLIT["bits"], SPLIT["group"], 128, 0.01)
    assert [res[r][:2] for r in range(world)] == [(0, 1472), (1472, 3000)]
    assert [res[r][2:4] for r in range(world)] == [(0, 32), (32, 96)]
    for r in range(world):
        assert np.array_equal(res[r][4], H1.numpy())
        for k, v in ref.items():
            assert np.array_equal(res[r][5][k], v.numpy()), k
