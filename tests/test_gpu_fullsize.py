"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (same batch budget).

Every query's count bound is compared bit for bit with the oracle's grid
reading; the pair sets of a seeded sample of query rows are compared with the
fp64 brute-force oracle (certain neighbours must all be present, nothing
outside the 1e-5 eps^2 boundary band may be added); every query must appear
in exactly one batch, and every row must contain its query."""
import numpy as np
import pytest

import datagen
import oracle
from conftest import golden_eps

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BENCH_BATCH_BYTES = 32 << 30
N_SAMPLE = 48


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_sampled_rows(cfg):
    _full_size(cfg, tensor=False)


@pytest.mark.parametrize("cfg", [2, 4])
def test_full_size_sampled_rows_tensor_cores(cfg):
    _full_size(cfg, tensor=True)


def _full_size(cfg, tensor):
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd

    x = datagen.generate(cfg)
    n = len(x)
    eps = golden_eps(cfg)
    sample = datagen.sample_queries(n, N_SAMPLE, seed=500 + cfg)
    j = edd.Join()
    j.set_refine(tensor)
    j.build(torch.from_numpy(x).cuda())
    counts = j.count(eps)
    want_bound = oracle.count_bound(x, eps)
    assert np.array_equal(counts.cpu().numpy(), want_bound)

    sample_d = torch.from_numpy(sample).cuda()
    seen = torch.zeros(n, dtype=torch.int32, device="cuda")
    got = {}
    pairs = [0]

    def take(b):
        q = torch.as_tensor(edd.DeviceArray(b.query_ids, (b.nq,), "<i8"), device="cuda")
        rp = torch.as_tensor(edd.DeviceArray(b.row_ptr, (b.nq + 1,), "<i8"), device="cuda")
        seen.index_add_(0, q, torch.ones_like(q, dtype=torch.int32))
        assert int((rp[1:] - rp[:-1]).min()) >= 1
        pairs[0] += b.nnz
        hit = torch.nonzero(torch.isin(q, sample_d)).flatten().cpu().numpy()
        if hit.size:
            cols = torch.as_tensor(edd.DeviceArray(b.cols, (b.nnz,), "<i4"), device="cuda")
            rph = rp.cpu().numpy()
            qh = q.cpu().numpy()
            for i in hit:
                got[int(qh[i])] = cols[rph[i]:rph[i + 1]].cpu().numpy()

    st = j.join(eps, BENCH_BATCH_BYTES, edd.HISS_OUT_CSR, False, take)
    j.close()
    assert int(seen.min()) == 1 and int(seen.max()) == 1
    assert st["pairs"] == pairs[0]
    assert sorted(got) == sorted(sample.tolist())
    want = oracle.row_sets(x, eps, sample)
    for k, q in enumerate(sample.tolist()):
        sure, band = want[k]
        g = set(got[q].tolist())
        assert len(g) == got[q].size
        assert q in g
        assert sure <= g, "cfg %d row %d misses %s" % (cfg, q, sorted(sure - g)[:5])
        assert g <= sure | band, "cfg %d row %d extra %s" % (cfg, q, sorted(g - sure - band)[:5])
        assert want_bound[q] >= len(sure)
