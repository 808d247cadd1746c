"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (same batch budget).

Every query's count bound is compared bit for bit with the oracle's grid
reading.  The rows checked against the fp64 brute-force oracle are 4,096
seeded random queries plus queries of the three cells with the most work
(|cell| x B_cell): every query of such a cell when the oracle's budget allows,
else whole query tiles spread over the cell, its first and its last (ragged)
tile included.  Those are the rows whose candidates span the most refinement
chunks.  For each row the oracle gives (count, sum of splitmix64(id) modulo
2^64, pairs inside the 1e-5 eps^2 band) without listing the pairs; the GPU's
CSR row gives the same digest.  A row whose digest differs is listed by the
oracle and may differ only by band pairs.  Every query must appear in exactly
one batch, every row must hold its query once, and no row may repeat an id."""
import numpy as np
import pytest

import datagen
import oracle
from conftest import golden_eps
from rowdigest import row_hash

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N_RANDOM = 4096
HEAVY_CELLS = 3
HEAVY_COORD_OPS = 3e11      # oracle budget for the heavy-cell rows: rows x n x d
_ORACLE_CACHE = {}


def _bench_batch_bytes():
    import bench
    return bench.DEFAULT_BATCH_BYTES


def _rows_to_check(x, eps, cfg):
    """Seeded random rows, then heavy-cell rows (original ids), and the
    oracle's count bounds."""
    n, d = x.shape
    g = oracle.grid(x, eps)
    bound = oracle.count_bound(x, eps, g)
    cs = g["cell_start"]
    size = np.diff(cs)
    work = size * bound[g["order"][cs[:-1]]]
    top = np.argsort(-work, kind="stable")[:HEAVY_CELLS]
    tq = 128 if d <= 64 else 64                    # the refinement's query tile
    per_cell = max(tq, int(HEAVY_COORD_OPS / (n * d) / HEAVY_CELLS))
    heavy = []
    for c in top:
        ids = g["order"][cs[c]:cs[c + 1]]          # the cell's queries in index order
        if ids.size <= per_cell:
            heavy.append(ids)
            continue
        ntile = (ids.size + tq - 1) // tq
        for t in np.unique(np.round(np.linspace(0, ntile - 1, max(2, per_cell // tq))).astype(np.int64)):
            heavy.append(ids[t * tq:(t + 1) * tq])
    rnd = datagen.sample_queries(n, N_RANDOM, seed=500 + cfg)
    rows = np.unique(np.concatenate([rnd] + heavy).astype(np.int64))
    return rows, bound


def _oracle_side(cfg):
    if cfg not in _ORACLE_CACHE:
        x = datagen.generate(cfg)
        eps = golden_eps(cfg)
        rows, bound = _rows_to_check(x, eps, cfg)
        cnt, h, band = oracle.rows_digest(x, eps, rows)
        _ORACLE_CACHE[cfg] = (x, eps, rows, bound, cnt, h, band)
    return _ORACLE_CACHE[cfg]


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_rows(cfg):
    _full_size(cfg, tensor=False)


@pytest.mark.parametrize("cfg", [2, 4])
def test_full_size_rows_tensor_cores(cfg):
    _full_size(cfg, tensor=True)


def _full_size(cfg, tensor):
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd

    x, eps, rows, want_bound, w_cnt, w_hash, w_band = _oracle_side(cfg)
    n = len(x)
    j = edd.Join()
    j.set_refine(tensor)
    j.build(torch.from_numpy(x).cuda())
    counts = j.count(eps)
    assert np.array_equal(counts.cpu().numpy(), want_bound)

    rows_d = torch.from_numpy(rows).cuda()
    seen = torch.zeros(n, dtype=torch.int32, device="cuda")
    got = {}
    pairs = [0]

    def take(b):
        q = torch.as_tensor(edd.DeviceArray(b.query_ids, (b.nq,), "<i8"), device="cuda")
        rp = torch.as_tensor(edd.DeviceArray(b.row_ptr, (b.nq + 1,), "<i8"), device="cuda")
        seen.index_add_(0, q, torch.ones_like(q, dtype=torch.int32))
        assert int((rp[1:] - rp[:-1]).min()) >= 1
        pairs[0] += b.nnz
        hit = torch.nonzero(torch.isin(q, rows_d)).flatten().cpu().numpy()
        if hit.size:
            cols = torch.as_tensor(edd.DeviceArray(b.cols, (b.nnz,), "<i4"), device="cuda")
            rph = rp.cpu().numpy()
            qh = q.cpu().numpy()
            for i in hit:
                got[int(qh[i])] = cols[rph[i]:rph[i + 1]].cpu().numpy()

    st = j.join(eps, _bench_batch_bytes(), edd.HISS_OUT_CSR, False, take)
    j.close()
    assert int(seen.min()) == 1 and int(seen.max()) == 1
    assert st["pairs"] == pairs[0]
    assert sorted(got) == rows.tolist()
    differ = []
    for k, q in enumerate(rows.tolist()):
        g = got[q]
        assert np.unique(g).size == g.size, "cfg %d row %d repeats an id" % (cfg, q)
        assert q in set(g.tolist())
        assert want_bound[q] >= w_cnt[k]
        if g.size != w_cnt[k] or row_hash(g) != int(w_hash[k]):
            assert w_band[k] > 0, "cfg %d row %d differs with no pair in the band" % (cfg, q)
            differ.append(q)
    # rows that differ are listed by the oracle: they may differ only by band pairs
    if differ:
        want = oracle.row_sets(x, eps, np.array(differ))
        for (sure, band), q in zip(want, differ):
            g = set(got[q].tolist())
            assert sure <= g, "cfg %d row %d misses %s" % (cfg, q, sorted(sure - g)[:5])
            assert g <= sure | band, "cfg %d row %d extra %s" % (cfg, q, sorted(g - sure - band)[:5])
