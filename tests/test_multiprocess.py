"""The benchmark's multi-rank path on CPU: two gloo ranks, each timing its
own replica of the workload; the job time is the slowest rank's and the
units are summed (no collective touches the join's data)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, units = bench.aggregate(1.5 + rank, 1000 * (rank + 1), dist, torch.device("cpu"))
    out.put((rank, t, units))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res == [(0, 2.5, 3000), (1, 2.5, 3000)]


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(2.0, 7) == (2.0, 7)
