"""Semi-join (Q distinct from D, RT-HiSS Section II-A) through the C ABI,
against the fp64 oracle: pair sets exact outside the 1e-5 eps^2 band, count
bounds bit-exact with the oracle's grid reading."""
import numpy as np
import pytest

import datagen
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _edd():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd
    return edd


def _check(xq, xd, eps, rows):
    want = oracle.semi_row_sets(xq, xd, eps)
    assert sorted(rows) == list(range(len(xq)))
    for r in range(len(xq)):
        sure, band = want[r]
        got = rows[r]
        g = set(got.tolist())
        assert len(g) == got.size
        assert sure <= g, "query %d misses %s" % (r, sorted(sure - g)[:5])
        assert g <= sure | band, "query %d extra %s" % (r, sorted(g - sure - band)[:5])


@pytest.mark.parametrize("cfg,nd,nq,eps", [(1, 3000, 1000, 0.6), (2, 5000, 800, 6.0), (5, 6000, 500, 0.9),
                                          (4, 2000, 300, 1.4)])
def test_semi_join_matches_oracle(cfg, nd, nq, eps):
    edd = _edd()
    xd = datagen.generate(cfg, n=nd)
    rng = np.random.default_rng(cfg)
    lo, hi = xd.min(0), xd.max(0)
    span = hi - lo
    xq = (lo - 0.2 * span + rng.random((nq, xd.shape[1])) * 1.4 * span).astype(np.float32)
    xq[: nq // 4] = xd[rng.choice(nd, nq // 4, replace=False)]          # some queries on data points
    j = edd.Join()
    j.build(torch.from_numpy(xd).cuda())
    qd = torch.from_numpy(xq).cuda()
    counts = j.count_queries(qd, eps).cpu().numpy()
    rows = j.join_queries_sets(qd, eps)
    st = j.stats()
    j.close()
    # the stage skip keeps every result pair's tile
    assert st["pairs"] <= st["candidates_refined"] <= st["candidates"]
    assert np.array_equal(counts, oracle.semi_count_bound(xq, xd, eps))
    _check(xq, xd, eps, rows)
    true = np.array([len(rows[r]) for r in range(nq)])
    assert np.all(counts >= true)


def test_semi_count_bound_hand_case_on_gpu():
    # the hand-computed bounds of tests/golden/semi_bound_hand.txt: queries one
    # and two cells outside D's grid, below and above, on every index dimension
    from test_oracle import semi_bound_hand_case
    edd = _edd()
    xq, xd, eps, want = semi_bound_hand_case()
    j = edd.Join()
    j.build(torch.from_numpy(xd).cuda())
    qd = torch.from_numpy(xq).cuda()
    counts = j.count_queries(qd, eps).cpu().numpy()
    rows = j.join_queries_sets(qd, eps)
    j.close()
    assert counts.tolist() == want
    _check(xq, xd, eps, rows)


def test_semi_join_with_queries_equal_to_data_is_self_join_and_self_join_still_works():
    edd = _edd()
    x = datagen.generate(1, n=2500)
    eps = 0.55
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    a = j.join_sets(eps)
    b = j.join_queries_sets(torch.from_numpy(x).cuda(), eps)
    c = j.join_sets(eps)
    j.close()
    for q in range(len(x)):
        assert np.array_equal(np.sort(a[q]), np.sort(b[q]))
        assert np.array_equal(np.sort(a[q]), np.sort(c[q]))


def test_semi_join_edge_cases_and_batching():
    edd = _edd()
    xd = datagen.generate(5, n=20000)
    j = edd.Join()
    j.build(torch.from_numpy(xd).cuda())
    empty = torch.zeros((0, xd.shape[1]), dtype=torch.float32, device="cuda")
    assert j.join_queries_sets(empty, 0.7) == {}
    far = torch.full((1, xd.shape[1]), 1e6, dtype=torch.float32, device="cuda")
    assert j.join_queries_sets(far, 0.7)[0].size == 0
    assert j.count_queries(far, 0.7).cpu().tolist() == [0]
    xq = datagen.generate(5, n=3000) + np.float32(0.01)
    qd = torch.from_numpy(xq).cuda()
    one = j.join_queries_sets(qd, 0.7)
    st1 = j.stats()
    many = j.join_queries_sets(qd, 0.7, batch_bytes=1 << 20)
    st2 = j.stats()
    j.close()
    assert st1["batches"] == 1 and st2["batches"] > 2
    assert st1["candidates_refined"] == st2["candidates_refined"]  # batching does not change the skip
    for r in range(len(xq)):
        assert np.array_equal(np.sort(one[r]), np.sort(many[r]))
    _check(xq[::29], xd, 0.7, {i: one[r] for i, r in enumerate(range(0, len(xq), 29))})
