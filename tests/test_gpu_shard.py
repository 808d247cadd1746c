"""The sharded self-join (hiss_join_shard): the shards of one join, run one
after another on one GPU, partition the queries and their union is the
join; each rank's share of the refinement units is about 1/nranks.  (Every
shard could run on its own GPU with its own context; nothing passes between
ranks.)"""
import numpy as np
import pytest

import datagen
from conftest import golden_eps

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _edd():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd
    return edd


@pytest.mark.parametrize("cfg,n,nranks,batch_bytes", [(1, None, 1, 0), (1, None, 2, 0), (1, None, 3, 0),
                                                     (1, None, 7, 0), (4, 6000, 3, 1 << 20), (3, 8000, 2, 1 << 20)])
def test_shards_partition_the_join(cfg, n, nranks, batch_bytes):
    # cfg 3 and 4 (d = 64, 128) run the chunk-by-chunk unit order, whose cell
    # runs are cut by shard and batch boundaries here
    edd = _edd()
    x = datagen.generate(cfg, n=n)
    eps = golden_eps(cfg) if n is None else float(np.float32(golden_eps(cfg) * 1.5))
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    full = j.join_sets(eps)
    total_units = j.stats()["refine_units"]
    seen = {}
    units = []
    for r in range(nranks):
        part = j.join_shard_sets(eps, r, nranks, batch_bytes)
        units.append(j.stats()["refine_units"])
        for q, cols in part.items():
            assert q not in seen, "query %d in two shards" % q
            seen[q] = cols
    j.close()
    assert set(seen) == set(full)
    for q, cols in full.items():
        assert sorted(seen[q].tolist()) == sorted(cols.tolist())
    assert sum(units) == total_units
    assert max(units) <= total_units / nranks + max(64, total_units // 50)


def test_shard_arguments():
    edd = _edd()
    j = edd.Join()
    j.build(torch.from_numpy(datagen.generate(1, n=500)).cuda())
    for rank, nranks in [(-1, 2), (2, 2), (0, 0)]:
        with pytest.raises(edd.HissError):
            j.join_shard(0.5, rank, nranks)
    j.close()
