"""Plant plausible mistakes in copies of the oracle's C source and check that
the pins catch every one.  The mutants are compiled on the CPU into temporary
libraries; the real oracle is untouched."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import datagen
import oracle
from conftest import read_golden

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "dropped_last_term": ("for (int k = 0; k < d; ++k)", "for (int k = 0; k < d - 1; ++k)"),
    "dropped_first_term": ("for (int k = 0; k < d; ++k)", "for (int k = 1; k < d; ++k)"),
    "sum_not_difference": ("(double)a[k] - (double)b[k]", "(double)a[k] + (double)b[k]"),
    "missing_square": ("s += t * t;", "s += t < 0 ? -t : t;"),
    "row_stride": ("x + j * (int64_t)d, d) <= hi", "x + j, d) <= hi"),
    "strict_rows": ("if (sqdist(q, x + j * (int64_t)d, d) <= hi)", "if (sqdist(q, x + j * (int64_t)d, d) < hi)"),
    "strict_counts": ("d, d) <= eps2)", "d, d) < eps2)"),
    "self_excluded": ("for (int64_t j = 0; j < n; ++j)\n            if (sqdist(q, x + j * (int64_t)d, d) <= hi)",
                      "for (int64_t j = 0; j < n; ++j)\n            if (j != rows[r] && sqdist(q, x + j * (int64_t)d, d) <= hi)"),
    "picker_keeps_self": ("if (j != i) buf[m++]", "buf[m++]"),
    "picker_off_by_one": ("const double a = pool[nq * K - 1], b = pool[nq * K];",
                          "const double a = pool[nq * K], b = pool[nq * K + 1];"),
    "digest_hash_shifted_id": ("h += splitmix64((uint64_t)j);", "h += splitmix64((uint64_t)j + 1);"),
    "digest_strict": ("if (s <= eps2) {", "if (s < eps2) {"),
    "digest_band_one_sided": ("if (s >= lo && s <= hi) ++b;", "if (s >= lo && s <= eps2) ++b;"),
    "picker_never_retries": ("if (!(b < kth[r])) { status = 1; break; }", "if (0) { status = 1; break; }"),
}


def _load(path):
    lib = ctypes.CDLL(path)
    i64, i32, f64, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
    lib.orc_rows_count.argtypes = [p, i64, i32, f64, f64, p, i64, p]
    lib.orc_counts.argtypes = [p, i64, i32, f64, p]
    lib.orc_pick_eps2.argtypes = [p, i64, i32, p, i64, i64, i64, p, p]
    lib.orc_pick_eps2.restype = ctypes.c_int
    lib.orc_rows_digest.argtypes = [p, i64, i32, f64, f64, p, i64, p, p, p]
    return lib


def _pin_cases():
    cases = []
    x = np.array([[0.0, 0.0], [3.0, 4.0]], dtype=np.float32)
    cases.append((x, 5.0, [2, 2]))
    x = np.zeros((4, 16), dtype=np.float32)
    x[1, :4] = 1.0
    x[2, 0] = 2.0
    x[3, :5] = 1.0
    cases.append((x, 2.0, [3, 4, 3, 2]))
    g = read_golden("fig3_relation.txt")
    pts = {int(t[1:]): [float(a) for a in v] for t, v in g if t.startswith("p") and t != "pair"}
    x = np.zeros((len(pts), 8), dtype=np.float32)
    for i, xy in pts.items():
        x[i, :2] = xy
    cases.append((x, 1.0, [2, 2, 2, 2, 1, 2, 2]))
    return cases


def _pins_hold(lib) -> bool:
    # row digest: the 3-4-5 pair lies exactly on eps (inside, and in the band)
    from rowdigest import splitmix64
    x = np.array([[0.0, 0.0], [3.0, 4.0], [10.0, 0.0]], dtype=np.float32)
    q = np.arange(3, dtype=np.int64)
    c, h, b = np.empty(3, np.int64), np.empty(3, np.uint64), np.empty(3, np.int64)
    lib.orc_rows_digest(x.ctypes.data, 3, 2, oracle.eps_squared(5.0), 1e-5, q.ctypes.data, 3, c.ctypes.data,
                        h.ctypes.data, b.ctypes.data)
    h01 = (int(splitmix64(0)) + int(splitmix64(1))) % (1 << 64)
    if c.tolist() != [2, 2, 1] or [int(v) for v in h] != [h01, h01, int(splitmix64(2))] or b.tolist() != [1, 1, 0]:
        return False
    # eps one float32 step below 5: the pair is just outside, still in the band
    e_lo = float(np.nextafter(np.float32(5.0), np.float32(0.0)))
    lib.orc_rows_digest(x.ctypes.data, 3, 2, oracle.eps_squared(e_lo), 1e-5, q.ctypes.data, 3, c.ctypes.data,
                        h.ctypes.data, b.ctypes.data)
    if c.tolist() != [1, 1, 1] or b.tolist() != [1, 1, 0]:
        return False
    for x, eps, want in _pin_cases():
        n, d = x.shape
        e2 = oracle.eps_squared(eps)
        q = np.arange(n, dtype=np.int64)
        c1 = np.empty(n, dtype=np.int64)
        lib.orc_rows_count(x.ctypes.data, n, d, e2, 0.0, q.ctypes.data, n, c1.ctypes.data)
        c2 = np.empty(n, dtype=np.int64)
        lib.orc_counts(x.ctypes.data, n, d, e2, c2.ctypes.data)
        if c1.tolist() != want or c2.tolist() != want:
            return False
    # epsilon picker against a pooled brute-force sort
    x = datagen.generate(1, n=600)
    q = datagen.sample_queries(len(x), 20, seed=3)
    a, b = ctypes.c_double(), ctypes.c_double()
    rc = lib.orc_pick_eps2(x.ctypes.data, len(x), x.shape[1], q.ctypes.data, q.size, 5, 599,
                           ctypes.byref(a), ctypes.byref(b))
    x64 = x.astype(np.float64)
    pooled = np.sort(np.concatenate([np.delete(((x64 - x64[i]) ** 2).sum(1), i) for i in q]))
    if not (rc == 0 and a.value == pooled[q.size * 5 - 1] and b.value == pooled[q.size * 5]):
        return False
    # the retry path: one dense query among sparse ones, M grown as oracle.pick_eps grows it
    rng = np.random.default_rng(21)
    x = np.concatenate([(rng.random((100, 3)) * 1e-3).astype(np.float32),
                        (rng.random((500, 3)) * 40.0 + 2.0).astype(np.float32)])
    q = np.r_[0, 100 + np.arange(9) * 50].astype(np.int64)
    m = 64
    while True:
        rc = lib.orc_pick_eps2(x.ctypes.data, len(x), x.shape[1], q.ctypes.data, q.size, 10, m,
                               ctypes.byref(a), ctypes.byref(b))
        if rc != 1 or m > 4 * len(x):
            break
        m *= 4
    x64 = x.astype(np.float64)
    pooled = np.sort(np.concatenate([np.delete(((x64 - x64[i]) ** 2).sum(1), i) for i in q]))
    return rc == 0 and a.value == pooled[q.size * 10 - 1] and b.value == pooled[q.size * 10]


def test_real_oracle_passes_mutant_pins(tmp_path):
    assert _pins_hold(_load(oracle.build()))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, name
    mutated = src.replace(old, new)
    c = tmp_path / ("m_%s.c" % name)
    so = tmp_path / ("m_%s.so" % name)
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", str(so), str(c)])
    assert not _pins_hold(_load(str(so))), "pins did not catch mutant %s" % name


# ---- kNN oracle: planted mistakes in copies of its Python definition ----------

def _knn_variant(kind):
    def knn(x, k, query_rows=None):
        x64 = np.asarray(x, np.float32).astype(np.float64)
        n = x64.shape[0]
        q = np.arange(n) if query_rows is None else np.asarray(query_rows)
        ids = np.empty((q.size, k), np.int64)
        d2 = np.empty((q.size, k))
        for r, i in enumerate(q.tolist()):
            s = ((x64 - x64[i]) ** 2).sum(axis=1)
            if kind == "abs_not_square":
                s = np.abs(x64 - x64[i]).sum(axis=1)
            if kind == "self_excluded":
                s[i] = np.inf
            tie = np.arange(n) if kind != "ties_by_higher_index" else -np.arange(n)
            order = np.lexsort((tie, s))
            if kind == "off_by_one":
                order = order[1:]
            order = order[:k]
            ids[r] = order
            d2[r] = s[order]
        return ids, d2
    return knn


def _knn_pins(knn):
    """The kNN pins of test_oracle.py, for a given implementation."""
    x = np.array([[0], [1], [3], [6], [10]], np.float32)
    ids, d2 = knn(x, 3)
    assert ids.tolist() == [[0, 1, 2], [1, 0, 2], [2, 1, 0], [3, 2, 4], [4, 3, 2]]
    assert d2.tolist() == [[0, 1, 9], [0, 1, 4], [0, 4, 9], [0, 9, 16], [0, 16, 49]]
    rng = np.random.default_rng(11)
    x = rng.integers(0, 4, size=(40, 3)).astype(np.float32)
    ids, _ = knn(x, 7)
    assert ids.tolist() == oracle.knn_py(x, 7)


def test_knn_pins_hold_for_the_oracle():
    _knn_pins(oracle.knn)


@pytest.mark.parametrize("kind", ["self_excluded", "ties_by_higher_index", "off_by_one", "abs_not_square"])
def test_knn_pins_catch_planted_mistakes(kind):
    with pytest.raises(AssertionError):
        _knn_pins(_knn_variant(kind))


# ---- semi-join count bound: planted mistakes in copies of its Python source ---

SEMI_BOUND_MUTANTS = {
    "stencil_radius_2": ("for dx, dy, dz in STENCIL:",
                         "for dx, dy, dz in [(a, b, c) for c in range(-2, 3) for b in range(-2, 3) "
                         "for a in range(-2, 3)]:"),
    "unsigned_clip": ("cq[:, k] = np.floor(u).astype(np.int64)",
                      "cq[:, k] = np.maximum(np.floor(u), 0).astype(np.int64)"),
    "truncate_not_floor": ("cq[:, k] = np.floor(u).astype(np.int64)", "cq[:, k] = u.astype(np.int64)"),
    "original_dimension_order": ('idx = g["perm"][: min(3, xd.shape[1])]', "idx = np.arange(min(3, xd.shape[1]))"),
    "origin_from_queries": ('- g["origin"][k]) / w', '- xq[:, idx[k]].min()) / w'),
}


def _semi_bound_variant(name):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.semi_count_bound))
    old, new = SEMI_BOUND_MUTANTS[name]
    assert old in src, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant %s>" % name, "exec"), ns)
    return ns["semi_count_bound"]


def test_semi_bound_pin_holds_for_the_oracle():
    from test_oracle import semi_bound_hand_case
    xq, xd, eps, want = semi_bound_hand_case()
    assert oracle.semi_count_bound(xq, xd, eps).tolist() == want


@pytest.mark.parametrize("name", sorted(SEMI_BOUND_MUTANTS))
def test_semi_bound_mutant_is_caught(name):
    from test_oracle import semi_bound_hand_case
    xq, xd, eps, want = semi_bound_hand_case()
    assert _semi_bound_variant(name)(xq, xd, eps).tolist() != want, "pin did not catch %s" % name
