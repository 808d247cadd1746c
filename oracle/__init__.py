"""Oracle for the exact epsilon self-join -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package never
imports the product path: the two share no code.  The only module both sides
use is ``datagen`` (seeded random inputs, none of the join's arithmetic).

What is here, each a plain restatement of RT-HiSS (Munugala & Gowanlock,
"RT-HiSS: Ray Tracing Accelerated High Dimensional Vector Similarity
Searches"):

* the join itself (Section II-A, "Problem Statement"): fp64 brute force in
  plain C (``oracle.c``), inclusive ``dist <= eps``, self pairs included;
* the variance order of the dimensions (Section IV-A);
* the three-dimensional grid index whose 27-cell stencil bounds each query's
  candidates (grid indexing of Section II-B1, with the Morton order of
  Section IV-C), written as numpy steps in the order the method takes them;
* the count bound of the first intersection test (Section IV-D);
* the stream compaction of the result mask (Section IV-F1, Fig. 5);
* a per-row digest (count, splitmix64 fingerprint, boundary-band count) of
  the join's rows, for comparing rows too large to list.

The grid, Morton key and count-bound functions define one reading of the
pages (the pages index with an RT-core BVH that this build replaces); each
reading is spelled out in the function's docstring.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib_handle = None

# Pairs whose squared distance lies within this relative band of eps^2 may be
# decided either way by a correct float32 implementation (see ``rows``).
BAND = 1e-5


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    stale = not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared",
                               "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        i64, i32, f64, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        lib.orc_rows_count.argtypes = [p, i64, i32, f64, f64, p, i64, p]
        lib.orc_rows_fill.argtypes = [p, i64, i32, f64, f64, p, i64, p, p, p, p]
        lib.orc_counts.argtypes = [p, i64, i32, f64, p]
        lib.orc_pick_eps2.argtypes = [p, i64, i32, p, i64, i64, i64, p, p]
        lib.orc_semi_count.argtypes = [p, i64, p, i64, i32, f64, f64, p]
        lib.orc_semi_fill.argtypes = [p, i64, p, i64, i32, f64, f64, p, p, p, p]
        lib.orc_rows_digest.argtypes = [p, i64, i32, f64, f64, p, i64, p, p, p]
        lib.orc_pick_eps2.restype = ctypes.c_int
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _points(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("points must be (n, d)")
    return x


def eps_squared(eps) -> float:
    """eps^2 in fp64 for the float32 eps the GPU receives."""
    e = float(np.float32(eps))
    return e * e


# --------------------------------------------------------------------------
# The join (Section II-A)
# --------------------------------------------------------------------------

def counts(x, eps) -> np.ndarray:
    """|N(i)| for every point i, self included (fp64 brute force)."""
    x = _points(x)
    out = np.empty(x.shape[0], dtype=np.int64)
    _lib().orc_counts(_ptr(x), x.shape[0], x.shape[1], eps_squared(eps), _ptr(out))
    return out


def rows(x, eps, query_rows, band: float = BAND):
    """Neighbour lists of the given query rows.

    Returns (row_ptr, cols, flag, dist2): for query r, cols[row_ptr[r]:
    row_ptr[r+1]] lists, in increasing order, every j with
    s(i, j) <= eps^2 (1 + band).  flag = 1 marks pairs in the boundary band
    |s - eps^2| <= band eps^2, which a float32 implementation may decide
    either way; flag = 0 marks certain neighbours.  With band = 0 the lists
    are exactly the rows of the definition.
    """
    x = _points(x)
    q = np.ascontiguousarray(query_rows, dtype=np.int64)
    lib = _lib()
    e2 = eps_squared(eps)
    cnt = np.empty(q.size, dtype=np.int64)
    lib.orc_rows_count(_ptr(x), x.shape[0], x.shape[1], e2, float(band), _ptr(q), q.size, _ptr(cnt))
    row_ptr = np.zeros(q.size + 1, dtype=np.int64)
    np.cumsum(cnt, out=row_ptr[1:])
    nnz = int(row_ptr[-1])
    cols = np.empty(max(nnz, 1), dtype=np.int32)
    flag = np.empty(max(nnz, 1), dtype=np.uint8)
    dist2 = np.empty(max(nnz, 1), dtype=np.float64)
    lib.orc_rows_fill(_ptr(x), x.shape[0], x.shape[1], e2, float(band), _ptr(q), q.size,
                      _ptr(row_ptr), _ptr(cols), _ptr(flag), _ptr(dist2))
    return row_ptr, cols[:nnz], flag[:nnz], dist2[:nnz]


def rows_digest(x, eps, query_rows, band: float = BAND):
    """Per query row i, without listing the pairs: (count, hash, band) with
    count = |{j : s(i, j) <= eps^2}| (the definition, no band), hash = the sum
    modulo 2^64 of splitmix64(j) over those j, and band = the number of j with
    |s(i, j) - eps^2| <= band eps^2.  Used to compare large rows."""
    x = _points(x)
    q = np.ascontiguousarray(query_rows, dtype=np.int64)
    cnt = np.empty(q.size, dtype=np.int64)
    h = np.empty(q.size, dtype=np.uint64)
    b = np.empty(q.size, dtype=np.int64)
    _lib().orc_rows_digest(_ptr(x), x.shape[0], x.shape[1], eps_squared(eps), float(band), _ptr(q), q.size,
                           _ptr(cnt), _ptr(h), _ptr(b))
    return cnt, h, b


def semi_rows(xq, xd, eps, band: float = BAND):
    """Semi-join rows (RT-HiSS Section II-A, Q distinct from D): for each
    query q_r, every j of D with s(q_r, p_j) <= eps^2 (1 + band), increasing;
    returns (row_ptr, cols, flag, dist2) as ``rows`` does."""
    xq = _points(xq)
    xd = _points(xd)
    if xq.shape[1] != xd.shape[1]:
        raise ValueError("queries and data must have the same dimension")
    lib = _lib()
    e2 = eps_squared(eps)
    cnt = np.empty(xq.shape[0], dtype=np.int64)
    lib.orc_semi_count(_ptr(xq), xq.shape[0], _ptr(xd), xd.shape[0], xd.shape[1], e2, float(band), _ptr(cnt))
    row_ptr = np.zeros(xq.shape[0] + 1, dtype=np.int64)
    np.cumsum(cnt, out=row_ptr[1:])
    nnz = int(row_ptr[-1])
    cols = np.empty(max(nnz, 1), dtype=np.int32)
    flag = np.empty(max(nnz, 1), dtype=np.uint8)
    dist2 = np.empty(max(nnz, 1), dtype=np.float64)
    lib.orc_semi_fill(_ptr(xq), xq.shape[0], _ptr(xd), xd.shape[0], xd.shape[1], e2, float(band), _ptr(row_ptr),
                      _ptr(cols), _ptr(flag), _ptr(dist2))
    return row_ptr, cols[:nnz], flag[:nnz], dist2[:nnz]


def semi_row_sets(xq, xd, eps, band: float = BAND):
    """Per query: (certain neighbours in D, band pairs) as two sets."""
    row_ptr, cols, flag, _ = semi_rows(xq, xd, eps, band)
    out = []
    for r in range(len(row_ptr) - 1):
        c = cols[row_ptr[r]:row_ptr[r + 1]]
        f = flag[row_ptr[r]:row_ptr[r + 1]]
        out.append((set(c[f == 0].tolist()), set(c[f == 1].tolist())))
    return out


def semi_brute_force_py(xq, xd, eps) -> list:
    """The semi-join definition as nested pure-Python loops (tiny inputs)."""
    xq = _points(xq)
    xd = _points(xd)
    e2 = eps_squared(eps)
    res = []
    for q in xq.tolist():
        row = set()
        for j, p in enumerate(xd.tolist()):
            s = 0.0
            for a, b in zip(q, p):
                t = a - b
                s += t * t
            if s <= e2:
                row.add(j)
        res.append(row)
    return res


def semi_count_bound(xq, xd, eps) -> np.ndarray:
    """Semi-join count bound: points of D in the 27 grid cells of D's grid
    around each query's cell (the query keyed into D's grid, cell coordinates
    taken as signed integers; a query more than one cell outside D's grid has
    no candidate)."""
    xq = _points(xq)
    xd = _points(xd)
    g = grid(xd, eps)
    idx = g["perm"][: min(3, xd.shape[1])]
    w = g["w"]
    cq = np.zeros((xq.shape[0], 3), dtype=np.int64)
    for k in range(idx.size):
        u = (xq[:, idx[k]].astype(np.float64) - g["origin"][k]) / w
        cq[:, k] = np.floor(u).astype(np.int64)
    ck = g["cell_key"]
    size = np.diff(g["cell_start"])
    table = {int(k): int(s) for k, s in zip(ck.tolist(), size.tolist())}
    out = np.zeros(xq.shape[0], dtype=np.int64)
    for r in range(xq.shape[0]):
        tot = 0
        for dx, dy, dz in STENCIL:
            a, b, c = cq[r, 0] + dx, cq[r, 1] + dy, cq[r, 2] + dz
            if min(a, b, c) < 0 or max(a, b, c) >= (1 << 21):
                continue
            tot += table.get(int(morton3(np.uint64(a), np.uint64(b), np.uint64(c))), 0)
        out[r] = tot
    return out


def row_sets(x, eps, query_rows, band: float = BAND):
    """Per query row: (certain neighbours, band pairs) as two Python sets."""
    row_ptr, cols, flag, _ = rows(x, eps, query_rows, band)
    out = []
    for r in range(len(row_ptr) - 1):
        c = cols[row_ptr[r]:row_ptr[r + 1]]
        f = flag[row_ptr[r]:row_ptr[r + 1]]
        out.append((set(c[f == 0].tolist()), set(c[f == 1].tolist())))
    return out


def brute_force_py(x, eps) -> list:
    """The definition as nested pure-Python loops (only for tiny inputs)."""
    x = _points(x)
    e2 = eps_squared(eps)
    pts = [[float(v) for v in row] for row in x]
    n, d = len(pts), x.shape[1]
    res = []
    for i in range(n):
        row = set()
        for j in range(n):
            s = 0.0
            for k in range(d):
                t = pts[i][k] - pts[j][k]
                s += t * t
            if s <= e2:
                row.add(j)
        res.append(row)
    return res


# --------------------------------------------------------------------------
# Epsilon picker (workload definition)
# --------------------------------------------------------------------------

def pick_eps(x, k_mean: int, qidx) -> dict:
    """eps such that the sampled queries have k_mean neighbours on average,
    self excluded.  With a, b the (nq*K)-th and (nq*K+1)-th smallest pooled
    squared distances, eps^2 = (a + b) / 2 and eps = float32(sqrt(eps^2))."""
    x = _points(x)
    q = np.ascontiguousarray(qidx, dtype=np.int64)
    a = ctypes.c_double()
    b = ctypes.c_double()
    m = max(4 * int(k_mean), 64)
    while True:
        rc = _lib().orc_pick_eps2(_ptr(x), x.shape[0], x.shape[1], _ptr(q), q.size, int(k_mean),
                                  m, ctypes.byref(a), ctypes.byref(b))
        if rc == 0:
            break
        if rc != 1:
            raise RuntimeError("orc_pick_eps2 failed (%d)" % rc)
        m *= 4
    e2 = 0.5 * (a.value + b.value)
    eps = np.float32(np.sqrt(e2))
    # eps is a float32: keep a <= eps^2 < b when a float32 lies in [sqrt(a), sqrt(b))
    zero = np.float32(0.0)
    while eps > 0 and float(eps) * float(eps) >= b.value:
        eps = np.nextafter(eps, zero)
    up = np.nextafter(eps, np.float32(np.inf))
    if float(eps) * float(eps) < a.value and float(up) * float(up) < b.value:
        eps = up
    return {"eps": float(eps), "eps_hex": float(eps).hex(), "a": a.value, "b": b.value,
            "eps2_mid": e2, "nq": int(q.size), "k": int(k_mean)}


# --------------------------------------------------------------------------
# Index: variance order (Section IV-A) and the 3-D grid with Morton order
# --------------------------------------------------------------------------

def dim_stats(x):
    """Per-dimension min, max and population variance, in fp64."""
    x64 = _points(x).astype(np.float64)
    return x64.min(axis=0), x64.max(axis=0), x64.var(axis=0)


def variance_order(var) -> np.ndarray:
    """Dimensions by decreasing variance; equal variances keep index order."""
    var = np.asarray(var, dtype=np.float64)
    return np.array(sorted(range(var.size), key=lambda k: (-var[k], k)), dtype=np.int64)


MORTON_BITS = 21      # bits per index dimension in a 63-bit key
SUB_BITS_MAX = 5      # sub-cell resolution used to order points inside a cell
CELL_MARGIN = 2.0 ** -10
EXTENT_BITS = 20


def morton3(f0, f1, f2) -> np.ndarray:
    """Interleave three coordinates: bit b of coordinate k goes to key bit
    3b + k (coordinate 0 in the lowest position)."""
    f = [np.asarray(v, dtype=np.uint64) for v in (f0, f1, f2)]
    key = np.zeros(f[0].shape, dtype=np.uint64)
    for b in range(MORTON_BITS):
        for k in range(3):
            bit = (f[k] >> np.uint64(b)) & np.uint64(1)
            key |= bit << np.uint64(3 * b + k)
    return key


def demorton3(key):
    key = np.asarray(key, dtype=np.uint64)
    out = [np.zeros(key.shape, dtype=np.uint64) for _ in range(3)]
    for b in range(MORTON_BITS):
        for k in range(3):
            bit = (key >> np.uint64(3 * b + k)) & np.uint64(1)
            out[k] |= bit << np.uint64(b)
    return out


def grid(x, eps) -> dict:
    """The grid index over the three highest-variance dimensions.

    Reading of the pages (grid indexing, Section II-B1; variance-ordered index
    dimensions, Section IV-A; Morton order of grouped points, Section IV-C):

    1. perm = variance order; the index dimensions are perm[0..2] (fewer if
       d < 3; a missing index coordinate is 0).
    2. origin m_k = min of index dimension k; E = largest extent max_k - m_k.
    3. cell side w = max(eps (1 + 2^-10), E 2^-20), in fp64 (w = 1 if that
       is 0).  w > eps, so a pair within eps differs by at most one cell on
       every index dimension: the 27 surrounding cells hold every neighbour.
    4. u_k = (x_k - m_k) / w in fp64; cell_k = floor(u_k).
    5. s = min(5, 21 - bits(largest cell coordinate)) sub-cell bits;
       fine_k = floor(u_k 2^s), so cell_k = fine_k >> s.
    6. key = Morton(fine_0, fine_1, fine_2); the cell key is key >> 3s (the
       Morton key of the cell coordinates).
    7. D' order = stable sort of the points by key (equal keys keep their
       original order); cells are the runs of equal cell keys in that order.
    """
    x = _points(x)
    n, d = x.shape
    x64 = x.astype(np.float64)
    mn, mx, var = dim_stats(x)
    perm = variance_order(var)
    idx = perm[: min(3, d)]
    origin = mn[idx]
    extent = float(np.max(mx[idx] - mn[idx])) if n else 0.0
    e = float(np.float32(eps))
    w = max(e * (1.0 + CELL_MARGIN), extent * 2.0 ** -EXTENT_BITS)
    if w == 0.0:
        w = 1.0
    cellmax = int(np.max(np.floor((mx[idx] - mn[idx]) / w))) if n else 0
    s = min(SUB_BITS_MAX, MORTON_BITS - cellmax.bit_length())
    fine = np.zeros((n, 3), dtype=np.uint64)
    for k in range(idx.size):
        u = (x64[:, idx[k]] - origin[k]) / w
        fine[:, k] = np.floor(u * float(2 ** s)).astype(np.uint64)
    key = morton3(fine[:, 0], fine[:, 1], fine[:, 2])
    order = np.argsort(key, kind="stable")
    ckey_sorted = key[order] >> np.uint64(3 * s)
    starts = np.flatnonzero(np.r_[True, ckey_sorted[1:] != ckey_sorted[:-1]]) if n else np.zeros(0, np.int64)
    cell_key = ckey_sorted[starts]
    cell_start = np.r_[starts, n].astype(np.int64)
    cell_of_sorted = np.repeat(np.arange(starts.size), np.diff(cell_start))
    return {"perm": perm, "origin": origin, "w": w, "sub_bits": s, "cellmax": cellmax,
            "fine": fine, "key": key, "order": order, "cell_key": cell_key,
            "cell_start": cell_start, "cell_of_sorted": cell_of_sorted}


STENCIL = [(dx, dy, dz) for dz in (-1, 0, 1) for dy in (-1, 0, 1) for dx in (-1, 0, 1)]


def stencil(g: dict) -> list:
    """For each cell (Morton order), the indices of the existing cells among
    its 27 surrounding cells (itself included), in the order dz, dy, dx with
    dz outermost."""
    ck = g["cell_key"]
    cx, cy, cz = [c.astype(np.int64) for c in demorton3(ck)]
    out = [[] for _ in range(ck.size)]
    lookup = {int(k): i for i, k in enumerate(ck.tolist())}
    for i in range(ck.size):
        for dx, dy, dz in STENCIL:
            a, b, c = cx[i] + dx, cy[i] + dy, cz[i] + dz
            if min(a, b, c) < 0:
                continue
            kk = int(morton3(np.uint64(a), np.uint64(b), np.uint64(c)))
            j = lookup.get(kk)
            if j is not None:
                out[i].append(j)
    return out


def count_bound(x, eps, g: dict | None = None) -> np.ndarray:
    """B_q: the number of points in the 27 cells around q's cell (q's own
    included), per point in original order.  This is the first intersection
    test's per-query candidate count (Section IV-D) for the grid index; it is
    an upper bound of |N(q)|."""
    x = _points(x)
    if g is None:
        g = grid(x, eps)
    ck = g["cell_key"]
    size = np.diff(g["cell_start"])
    cx, cy, cz = [c.astype(np.int64) for c in demorton3(ck)]
    bound = np.zeros(ck.size, dtype=np.int64)
    for dx, dy, dz in STENCIL:
        a, b, c = cx + dx, cy + dy, cz + dz
        ok = (a >= 0) & (b >= 0) & (c >= 0)
        nk = morton3(np.where(ok, a, 0), np.where(ok, b, 0), np.where(ok, c, 0))
        pos = np.searchsorted(ck, nk)
        posc = np.minimum(pos, max(ck.size - 1, 0))
        hit = ok & (pos < ck.size) & (ck[posc] == nk)
        bound += np.where(hit, size[posc], 0)
    per_sorted = bound[g["cell_of_sorted"]]
    out = np.empty(x.shape[0], dtype=np.int64)
    out[g["order"]] = per_sorted
    return out


# --------------------------------------------------------------------------
# Result mask compaction (Section IV-F1, Fig. 5)
# --------------------------------------------------------------------------

def compact_mask(bits) -> np.ndarray:
    """Positions of the ones of a 0/1 result mask, in increasing order."""
    b = np.asarray(bits).astype(bool)
    return np.array([i for i in range(b.size) if b[i]], dtype=np.int64)


# --------------------------------------------------------------------------
# Exact k nearest neighbours (RT-HiSS Section VI, "exact kNN" built on the
# epsilon join by growing eps)
# --------------------------------------------------------------------------

def knn(x, k: int, query_rows=None):
    """The k nearest points of each query row, fp64 brute force.

    Reading of the pages: RT-HiSS names exact kNN as a use of the epsilon
    join (repeat the join with a growing eps for the queries that have fewer
    than k neighbours, then keep the k nearest).  The result is the plain
    definition: for query i, the k points j (the point itself included, at
    distance 0) with the smallest squared distance s(i, j); equal distances
    are ordered by the lower index.  Returns (ids int64 [q, k], dist2 float64
    [q, k]), each row in increasing (s, j) order.
    """
    x = _points(x)
    n = x.shape[0]
    q = np.arange(n) if query_rows is None else np.asarray(query_rows, dtype=np.int64)
    if not 1 <= k <= n:
        raise ValueError("k must be in [1, n]")
    x64 = x.astype(np.float64)
    ids = np.empty((q.size, k), dtype=np.int64)
    d2 = np.empty((q.size, k), dtype=np.float64)
    for r, i in enumerate(q.tolist()):
        s = ((x64 - x64[i]) ** 2).sum(axis=1)
        order = np.lexsort((np.arange(n), s))[:k]  # by s, then by index
        ids[r] = order
        d2[r] = s[order]
    return ids, d2


def knn_py(x, k: int) -> list:
    """Pure-Python kNN for tiny inputs (a second, independent restatement
    used to pin ``knn``)."""
    pts = [[float(v) for v in row] for row in _points(x)]
    out = []
    for i, a in enumerate(pts):
        cand = []
        for j, b in enumerate(pts):
            s = 0.0
            for u, v in zip(a, b):
                s += (u - v) * (u - v)
            cand.append((s, j))
        cand.sort()
        out.append([j for _, j in cand[:k]])
    return out
