"""Pins for the CPU oracle: hand-computed cases, the pages' worked examples,
invariants of the definition and brute force on tiny inputs.  CPU only."""
import ctypes

import numpy as np
import pytest

import datagen
import oracle
from conftest import read_golden


def _sets(x, eps):
    row_ptr, cols, _, _ = oracle.rows(x, eps, np.arange(len(x)), band=0.0)
    return [set(cols[row_ptr[i]:row_ptr[i + 1]].tolist()) for i in range(len(x))]


def test_three_four_five_inclusive():
    x = np.array([[0.0, 0.0], [3.0, 4.0]], dtype=np.float32)
    assert _sets(x, 5.0) == [{0, 1}, {0, 1}]          # dist == eps is a neighbour
    below = np.nextafter(np.float32(5.0), np.float32(0.0))
    assert _sets(x, below) == [{0}, {1}]
    assert list(oracle.counts(x, 5.0)) == [2, 2]


def test_sphere_16d_exact_boundary():
    x = np.zeros((4, 16), dtype=np.float32)
    x[1, :4] = 1.0            # |x1 - x0|^2 = 4 = eps^2
    x[2, 0] = 2.0             # |x2 - x0|^2 = 4; |x2 - x1|^2 = 1 + 3 = 4
    x[3, :5] = 1.0            # |x3 - x0|^2 = 5; |x3 - x1|^2 = 1; |x3 - x2|^2 = 1 + 4 = 5
    got = _sets(x, 2.0)
    assert got == [{0, 1, 2}, {0, 1, 2, 3}, {0, 1, 2}, {1, 3}]


def test_fig3_relation():
    g = read_golden("fig3_relation.txt")
    eps = float([v for t, v in g if t == "eps"][0][0])
    d = int([v for t, v in g if t == "d"][0][0])
    pts = {int(t[1:]): [float(a) for a in v] for t, v in g if t.startswith("p") and t != "pair"}
    x = np.zeros((len(pts), d), dtype=np.float32)
    for i, xy in pts.items():
        x[i, :2] = xy
    want = [{i} for i in range(len(pts))]
    for t, v in g:
        if t == "pair":
            i, j = int(v[0]), int(v[1])
            want[i].add(j)
            want[j].add(i)
    assert _sets(x, eps) == want
    assert oracle.brute_force_py(x, eps) == want


def test_fig5_compaction():
    g = dict(read_golden("fig5_mask.txt"))
    mask = [int(v) for v in g["mask"]]
    assert oracle.compact_mask(mask).tolist() == [int(v) for v in g["positions"]]


@pytest.mark.parametrize("d", [1, 3, 7, 16])
def test_brute_force_matches_plain_loops(d):
    rng = np.random.default_rng(100 + d)
    x = rng.random((150, d)).astype(np.float32)
    x[10] = x[3]                              # a duplicate pair
    eps = float(np.sqrt(d) * 0.25)
    assert _sets(x, eps) == oracle.brute_force_py(x, eps)


def test_invariants_symmetry_self_monotone():
    x = datagen.generate(1, n=1500)
    eps_small, eps_big = 0.45, 0.55
    s1 = _sets(x, eps_small)
    s2 = _sets(x, eps_big)
    for i, row in enumerate(s1):
        assert i in row                                     # self included
        for j in row:
            assert i in s1[j]                               # symmetry
        assert row <= s2[i]                                 # monotone in eps
    c = oracle.counts(x, eps_small)
    assert c.tolist() == [len(r) for r in s1]


def test_duplicates_single_point_and_eps_zero():
    x = np.array([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0], [1.0, 2.0, 3.5]], dtype=np.float32)
    assert _sets(x, 0.0) == [{0, 1}, {0, 1}, {2}]
    assert _sets(x[:1], 0.0) == [{0}]


def test_band_flags():
    x = np.zeros((3, 2), dtype=np.float32)
    x[1, 0] = 1.0
    x[2, 0] = np.float32(1.0 + 2e-6)          # s - eps^2 ~ 4e-6 eps^2: inside the band
    row_ptr, cols, flag, dist2 = oracle.rows(x, 1.0, [0])
    assert cols.tolist() == [0, 1, 2]
    assert flag.tolist() == [0, 1, 1]
    assert dist2[1] == 1.0


def test_pick_eps_sample_identity():
    x = datagen.generate(1, n=3000)
    q = datagen.sample_queries(len(x), 100, seed=7)
    k = 10
    r = oracle.pick_eps(x, k, q)
    # brute force: pool every (query, other point) squared distance, sort
    x64 = x.astype(np.float64)
    pooled = []
    for i in q:
        s = ((x64 - x64[i]) ** 2).sum(axis=1)
        pooled.append(np.delete(s, i))
    pooled = np.sort(np.concatenate(pooled))
    assert r["a"] == pooled[len(q) * k - 1]
    assert r["b"] == pooled[len(q) * k]
    e2 = oracle.eps_squared(r["eps"])
    assert int(np.sum(pooled <= e2)) == len(q) * k            # mean K, self excluded


def _retry_instance():
    """One dense query among sparse ones: its first M = 64 kept distances all
    lie below the pooled (nq K + 1)-th value, so the picker must retry with a
    larger M before its answer is exact (RT-HiSS Section V-B defines the
    selectivity the picker targets)."""
    rng = np.random.default_rng(21)
    dense = (rng.random((100, 3)) * 1e-3).astype(np.float32)            # 100 points within 1e-3
    sparse = (rng.random((500, 3)) * 40.0 + 2.0).astype(np.float32)     # far from the dense ball
    x = np.concatenate([dense, sparse])
    q = np.r_[0, 100 + np.arange(9) * 50].astype(np.int64)              # 1 dense query, 9 sparse
    return x, q, 10


def _pooled(x, q):
    x64 = x.astype(np.float64)
    return np.sort(np.concatenate([np.delete(((x64 - x64[i]) ** 2).sum(1), i) for i in q]))


def test_pick_eps_retry_path():
    x, q, k = _retry_instance()
    # the first attempt keeps M = max(4 K, 64) distances per query and must ask for more
    a, b = ctypes.c_double(), ctypes.c_double()
    rc = oracle._lib().orc_pick_eps2(x.ctypes.data, len(x), x.shape[1], q.ctypes.data, q.size, k, 64,
                                     ctypes.byref(a), ctypes.byref(b))
    assert rc == 1
    pooled = _pooled(x, q)
    assert a.value != pooled[q.size * k - 1]          # the truncated pool alone would be wrong
    r = oracle.pick_eps(x, k, q)
    assert r["a"] == pooled[q.size * k - 1]
    assert r["b"] == pooled[q.size * k]
    e2 = oracle.eps_squared(r["eps"])
    assert int(np.sum(pooled <= e2)) == q.size * k


def test_pick_eps_many_equal_distances():
    # 20 groups of 20 equal points: a = b; the picker still returns a <= eps^2
    x = np.zeros((400, 2), dtype=np.float32)
    x[:, 0] = np.repeat(np.arange(20), 20).astype(np.float32)
    q = np.arange(0, 400, 40)
    r = oracle.pick_eps(x, 30, q)
    pooled = _pooled(x, q)
    assert r["a"] == pooled[q.size * 30 - 1] and r["b"] == pooled[q.size * 30]


# ---------------- index pins -----------------------------------------------

def test_morton_known_values_and_roundtrip():
    assert int(oracle.morton3(1, 0, 0)) == 1
    assert int(oracle.morton3(0, 1, 0)) == 2
    assert int(oracle.morton3(0, 0, 1)) == 4
    assert int(oracle.morton3(3, 3, 3)) == 63
    assert int(oracle.morton3(2, 0, 0)) == 8
    top = (1 << 21) - 1
    assert int(oracle.morton3(top, top, top)) == (1 << 63) - 1
    rng = np.random.default_rng(3)
    f = rng.integers(0, 1 << 21, size=(3, 500)).astype(np.uint64)
    back = oracle.demorton3(oracle.morton3(*f))
    for k in range(3):
        assert np.array_equal(back[k], f[k])


def test_dim_stats_closed_form_and_ties():
    x = np.zeros((4, 4), dtype=np.float32)
    x[:, 0] = [0, 2, 0, 2]        # variance 1
    x[:, 1] = [1, 1, 1, 1]        # variance 0
    x[:, 2] = [0, 4, 0, 4]        # variance 4
    x[:, 3] = [5, 3, 5, 3]        # variance 1 (ties with dim 0)
    mn, mx, var = oracle.dim_stats(x)
    assert var.tolist() == [1.0, 0.0, 4.0, 1.0]
    assert mn.tolist() == [0, 1, 0, 3] and mx.tolist() == [2, 1, 4, 5]
    assert oracle.variance_order(var).tolist() == [2, 0, 3, 1]


def test_grid_hand_case():
    # index dims: variance order puts dim 1 first, then 0, then 2
    x = np.array([[0.0, 0.0, 0.0, 9.0],
                  [0.5, 1.5, 0.0, 9.0],
                  [0.5, 3.5, 0.0, 9.0],
                  [0.5, 3.6, 0.0, 9.0],
                  [0.0, 9.0, 0.1, 9.0]], dtype=np.float32)
    g = oracle.grid(x, 1.0)
    assert g["perm"][:3].tolist() == [1, 0, 2]
    w = 1.0 * (1 + 2 ** -10)
    assert g["w"] == w
    cells = (g["fine"] >> np.uint64(g["sub_bits"])).astype(int)
    assert cells[:, 0].tolist() == [0, 1, 3, 3, 8]          # floor(x_1 / w)
    assert cells[:, 1].tolist() == [0, 0, 0, 0, 0]
    b = oracle.count_bound(x, 1.0, g)
    # cells on dim 1: {0: p0}, {1: p1}, {3: p2, p3}, {8: p4}
    assert b.tolist() == [2, 2, 2, 2, 1]


def test_stencil_matches_brute_force_adjacency():
    x = datagen.generate(5, n=4000)
    g = oracle.grid(x, 0.6)
    st = oracle.stencil(g)
    cx, cy, cz = [c.astype(int) for c in oracle.demorton3(g["cell_key"])]
    C = g["cell_key"].size
    for i in range(0, C, max(1, C // 60)):
        want = [j for j in range(C)
                if max(abs(cx[i] - cx[j]), abs(cy[i] - cy[j]), abs(cz[i] - cz[j])) <= 1]
        assert sorted(st[i]) == want
        # order: dz outermost, then dy, then dx
        keys = [(cz[j] - cz[i], cy[j] - cy[i], cx[j] - cx[i]) for j in st[i]]
        assert keys == sorted(keys)


@pytest.mark.parametrize("cfg,n,eps", [(1, 2000, 0.45), (2, 3000, 6.0), (5, 3000, 0.9)])
def test_count_bound_covers_true_count(cfg, n, eps):
    x = datagen.generate(cfg, n=n)
    b = oracle.count_bound(x, eps)
    c = oracle.counts(x, eps)
    assert np.all(b >= c)
    assert np.all(c >= 1)


def test_grid_order_is_stable_sort_by_key():
    x = datagen.generate(2, n=1000)
    g = oracle.grid(x, 5.0)
    key = g["key"].tolist()
    want = sorted(range(len(key)), key=lambda i: (key[i], i))
    assert g["order"].tolist() == want
    # points of one cell are contiguous in D' order
    ck = (g["key"][g["order"]] >> np.uint64(3 * g["sub_bits"])).tolist()
    seen, last = set(), None
    for v in ck:
        if v != last:
            assert v not in seen
            seen.add(v)
            last = v


def test_grid_neighbours_within_one_cell():
    x = datagen.generate(1, n=800)
    eps = 0.5
    g = oracle.grid(x, eps)
    cells = (g["fine"] >> np.uint64(g["sub_bits"])).astype(np.int64)
    for i, row in enumerate(_sets(x, eps)):
        for j in row:
            assert np.max(np.abs(cells[i] - cells[j])) <= 1


# ---------------- semi-join (Q distinct from D) -----------------------------

def test_semi_join_hand_case():
    xd = np.array([[0.0, 0.0], [3.0, 4.0], [10.0, 0.0]], dtype=np.float32)
    xq = np.array([[0.0, 0.0], [6.0, 8.0], [13.0, 4.0], [50.0, 50.0]], dtype=np.float32)
    row_ptr, cols, _, _ = oracle.semi_rows(xq, xd, 5.0, band=0.0)
    rows = [sorted(cols[row_ptr[i]:row_ptr[i + 1]].tolist()) for i in range(4)]
    assert rows == [[0, 1], [1], [2], []]          # |(6,8)-(3,4)| = 5 inclusive; (13,4)-(10,0) = 5
    assert oracle.semi_brute_force_py(xq, xd, 5.0) == [{0, 1}, {1}, {2}, set()]


def test_splitmix64_published_outputs():
    from rowdigest import splitmix64
    assert int(splitmix64(0)) == 0xE220A8397B1DCDAF                   # seed 0, first output
    # seed 1234567: first and second outputs (the second is seeded one golden step on)
    assert int(splitmix64(1234567)) == 6457827717110365317
    assert int(splitmix64(1234567 + 0x9E3779B97F4A7C15)) == 3203168211198807973


def test_rows_digest_hand_case():
    from rowdigest import splitmix64
    x = np.array([[0.0, 0.0], [3.0, 4.0], [10.0, 0.0]], dtype=np.float32)
    c, h, b = oracle.rows_digest(x, 5.0, [0, 1, 2])
    h01 = (int(splitmix64(0)) + int(splitmix64(1))) % (1 << 64)
    assert c.tolist() == [2, 2, 1]
    assert [int(v) for v in h] == [h01, h01, int(splitmix64(2))]
    assert b.tolist() == [1, 1, 0]                     # the 3-4-5 pair sits exactly on eps
    # eps one float32 step below 5: the pair is just outside eps, still in the band
    c, h, b = oracle.rows_digest(x, float(np.nextafter(np.float32(5.0), np.float32(0.0))), [0, 1, 2])
    assert c.tolist() == [1, 1, 1] and b.tolist() == [1, 1, 0]
    assert [int(v) for v in h] == [int(splitmix64(0)), int(splitmix64(1)), int(splitmix64(2))]


def test_rows_digest_matches_listed_rows():
    from rowdigest import row_hash
    x = datagen.generate(2, n=3000)
    q = datagen.sample_queries(len(x), 200, seed=4)
    eps = oracle.pick_eps(x, 20, q)["eps"]
    c, h, b = oracle.rows_digest(x, eps, q)
    row_ptr, cols, flag, dist2 = oracle.rows(x, eps, q)
    e2 = oracle.eps_squared(eps)
    for r in range(q.size):
        sl = slice(row_ptr[r], row_ptr[r + 1])
        inside = cols[sl][dist2[sl] <= e2]
        assert c[r] == inside.size
        assert int(h[r]) == row_hash(inside)
        assert b[r] == int(flag[sl].sum())


def semi_bound_hand_case():
    """The hand-computed semi-join count bounds of tests/golden/semi_bound_hand.txt."""
    g = read_golden("semi_bound_hand.txt")
    xd = np.array([[float(v) for v in vals] for t, vals in g if t == "d"], np.float32)
    xq = np.array([[float(v) for v in vals[:3]] for t, vals in g if t == "q"], np.float32)
    want = [int(vals[3]) for t, vals in g if t == "q"]
    eps = float([vals for t, vals in g if t == "eps"][0][0])
    return xq, xd, eps, want


def test_semi_count_bound_hand_case():
    # queries inside, one and two cells outside D's grid on each index
    # dimension, below and above, on a variance order that is not the identity
    xq, xd, eps, want = semi_bound_hand_case()
    assert oracle.grid(xd, eps)["perm"].tolist() == [1, 2, 0]
    assert oracle.semi_count_bound(xq, xd, eps).tolist() == want


def test_semi_join_with_q_equal_d_is_self_join():
    x = datagen.generate(1, n=600)
    a = oracle.semi_rows(x, x, 0.5, band=0.0)
    b = oracle.rows(x, 0.5, np.arange(len(x)), band=0.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_semi_join_matches_plain_loops_and_bound_covers():
    rng = np.random.default_rng(5)
    xd = rng.random((300, 5)).astype(np.float32)
    xq = (rng.random((120, 5)) * 1.4 - 0.2).astype(np.float32)   # some queries outside D's box
    eps = 0.35
    row_ptr, cols, _, _ = oracle.semi_rows(xq, xd, eps, band=0.0)
    got = [set(cols[row_ptr[i]:row_ptr[i + 1]].tolist()) for i in range(len(xq))]
    assert got == oracle.semi_brute_force_py(xq, xd, eps)
    bound = oracle.semi_count_bound(xq, xd, eps)
    assert all(bound[i] >= len(got[i]) for i in range(len(xq)))


# ---- exact kNN oracle --------------------------------------------------------

def test_knn_hand_case_1d_with_tie():
    # points 0, 1, 3, 6, 10 on a line; k = 3, self first; point 2 (x = 3) is
    # at 9 from both point 0 and point 3: the lower index wins
    x = np.array([[0], [1], [3], [6], [10]], np.float32)
    ids, d2 = oracle.knn(x, 3)
    assert ids.tolist() == [[0, 1, 2], [1, 0, 2], [2, 1, 0], [3, 2, 4], [4, 3, 2]]
    assert d2.tolist() == [[0, 1, 9], [0, 1, 4], [0, 4, 9], [0, 9, 16], [0, 16, 49]]


def test_knn_duplicates_ordered_by_index():
    x = np.zeros((6, 3), np.float32)
    x[4] = [1, 0, 0]
    ids, d2 = oracle.knn(x, 5)
    for i in range(6):
        if i == 4:
            assert ids[i].tolist() == [4, 0, 1, 2, 3]
        else:
            assert ids[i].tolist() == [0, 1, 2, 3, 5]
            assert np.all(d2[i] == 0)


def test_knn_matches_pure_python_loops():
    rng = np.random.default_rng(11)
    x = rng.integers(0, 4, size=(40, 3)).astype(np.float32)  # many exact ties
    ids, _ = oracle.knn(x, 7)
    assert ids.tolist() == oracle.knn_py(x, 7)


def test_knn_consistent_with_join_rows():
    x = datagen.generate(2, n=800)
    k = 10
    ids, d2 = oracle.knn(x, k)
    for i in range(0, 800, 37):
        r = float(np.sqrt(d2[i, -1]))
        rp, cols, _, _ = oracle.rows(x, np.float32(r) * np.float32(1.0001), [i], band=0.0)
        assert set(ids[i].tolist()) <= set(cols.tolist())
        assert len(cols) >= k


def test_knn_matches_sklearn_brute_force():
    nn = pytest.importorskip("sklearn.neighbors")
    x = datagen.generate(4, n=500)
    ids, d2 = oracle.knn(x, 8)
    ref = nn.NearestNeighbors(n_neighbors=8, algorithm="brute").fit(x.astype(np.float64))
    dist, rid = ref.kneighbors(x.astype(np.float64))
    assert np.array_equal(ids, rid)
    assert np.allclose(d2, dist ** 2, rtol=1e-9, atol=1e-12)
