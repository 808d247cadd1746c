"""Exact kNN by epsilon expansion (hiss_knn) on the GPU against the fp64
oracle.  The GPU orders by float32 squared distance, so a neighbour may
differ from the oracle's only where its exact squared distance is within the
float32 band of the k-th one; everything clearly closer must be present,
nothing clearly farther may be."""
import numpy as np
import pytest

import datagen
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BAND = 1e-5


def _edd():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd
    return edd


def _knn(x, k, eps0=0.0, tensor=False):
    edd = _edd()
    j = edd.Join()
    j.set_refine(tensor)
    j.build(torch.from_numpy(np.ascontiguousarray(x)).cuda())
    ids, d2 = j.knn(k, eps0)
    j.close()
    return ids.cpu().numpy(), d2.cpu().numpy()


def _check(x, k, ids, d2, qsel=None):
    n = len(x)
    qsel = np.arange(n) if qsel is None else np.asarray(qsel)
    want_ids, want_d2 = oracle.knn(x, k, qsel)
    x64 = x.astype(np.float64)
    for r, i in enumerate(qsel.tolist()):
        got = ids[i]
        assert len(set(got.tolist())) == k, "duplicate id in row %d" % i
        assert np.all(np.diff(d2[i]) >= 0), "row %d not sorted" % i
        rk = want_d2[r, -1]
        exact = ((x64[got] - x64[i]) ** 2).sum(axis=1)
        lo, hi = rk * (1 - BAND) - 1e-30, rk * (1 + BAND) + 1e-30
        sure = set(want_ids[r][want_d2[r] < lo].tolist())
        assert sure <= set(got.tolist()), "row %d misses %s" % (i, sorted(sure - set(got.tolist()))[:5])
        assert np.all(exact <= hi), "row %d holds a farther point" % i
        assert np.allclose(d2[i], exact, rtol=2e-6 * x.shape[1], atol=1e-30)
        assert got[0] == i or exact[0] == 0.0  # the point itself (or a duplicate) comes first


@pytest.mark.parametrize("cfg,n,k", [(1, 4000, 16), (2, 5000, 10), (3, 4000, 32), (4, 3000, 8), (5, 6000, 50)])
def test_knn_small_workloads(cfg, n, k):
    x = datagen.generate(cfg, n=n)
    ids, d2 = _knn(x, k)
    _check(x, k, ids, d2)


def test_knn_k_one_and_k_n_and_duplicates():
    x = datagen.generate(1, n=300)
    x[50:60] = x[5]
    ids, d2 = _knn(x, 1)
    assert np.all(d2[:, 0] == 0)
    for i in range(300):
        want = 5 if (i == 5 or 50 <= i < 60) else i
        assert ids[i, 0] == want
    ids, d2 = _knn(x, 300)
    _check(x, 300, ids, d2, qsel=np.arange(0, 300, 7))


def test_knn_outliers_need_many_rounds():
    # a tight cluster plus far outliers: the outliers need eps to grow far
    rng = np.random.default_rng(8)
    x = rng.normal(0, 0.01, (2000, 6)).astype(np.float32)
    x[:5] += np.float32(50.0)
    x[5:8] -= np.float32(200.0)
    ids, d2 = _knn(x, 12, eps0=0.001)
    _check(x, 12, ids, d2, qsel=np.r_[np.arange(0, 20), np.arange(100, 2000, 97)])


def test_knn_tensor_refinement_and_given_eps0():
    x = datagen.generate(2, n=4000)
    ids, d2 = _knn(x, 20, eps0=1.0, tensor=True)
    _check(x, 20, ids, d2, qsel=np.arange(0, 4000, 13))
