"""The sharded self-join across processes: two ranks (separate processes,
each with its own context on cuda:0, as each would have on its own GPU) build
the same index from the same points, join their shard (hiss_join_shard) and
gather their rows over gloo.  Together the shards must be the whole join,
each query in exactly one shard, and the benchmark's aggregate over the same
process group must give the slower rank's time and the summed pairs.  The
ranks' kernels never wait on one another: the only exchange is on the host,
after the joins."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import __graft_entry__
        __graft_entry__.build()
        import datagen
        import exact_dimensional_distance_gb300 as edd
        from conftest import golden_eps
        torch.cuda.set_device(0)
        x = datagen.generate(2, n=20000)
        eps = golden_eps(2) * 0.5
        j = edd.Join()
        j.build(torch.from_numpy(x).cuda())
        rows = j.join_shard_sets(eps, rank, world)
        st = j.stats()
        mine = {q: np.sort(c).tolist() for q, c in rows.items()}
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        import bench
        t, units = bench.aggregate(1.0 + rank, st["pairs"], dist, torch.device("cpu"))
        full = None
        if rank == 0:
            full = {q: np.sort(c).tolist() for q, c in j.join_sets(eps).items()}
        j.close()
        out.put((rank, gathered if rank == 0 else None, full, t, units, st["pairs"]))
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report instead of hanging the parent
        out.put((rank, "error", repr(e), None, None, None))
        raise


def test_two_ranks_shard_one_join_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r = q.get(timeout=600)
        assert r[1] != "error", r
        res[r[0]] = r
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    gathered, full = res[0][1], res[0][2]
    seen = {}
    for rank, shard in enumerate(gathered):
        for qid, cols in shard.items():
            assert qid not in seen, "query %d in shards %d and %d" % (qid, seen[qid], rank)
            seen[qid] = rank
            assert cols == full[qid]
    assert set(seen) == set(full)
    assert all(len(s) > 0 for s in gathered)
    # the benchmark's aggregate over the same group: slower time, summed pairs
    total = sum(res[r][5] for r in res)
    assert all(res[r][3] == 2.0 and res[r][4] == total for r in res)
    assert total == sum(len(c) for c in full.values())
