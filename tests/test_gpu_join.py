"""Parity of the CUDA join with the fp64 oracle, through the C ABI.

Pair sets must match the oracle exactly except for pairs whose squared
distance lies within 1e-5 eps^2 of eps^2 (oracle.BAND): a float32 sum of d
squared differences carries a relative error of at most about (d + 2) 2^-24,
below 1e-5 for the dimensions tested here.  Index and count results are
integers and must match bit for bit."""
import numpy as np
import pytest

import datagen
import oracle
from conftest import golden_eps

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _edd():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd
    return edd


def _join(x, eps, batch_bytes=0):
    edd = _edd()
    j = edd.Join()
    j.build(torch.from_numpy(np.ascontiguousarray(x)).cuda())
    counts = j.count(eps).cpu().numpy()
    rows = j.join_sets(eps, batch_bytes)
    st = j.stats()
    j.close()
    return rows, counts, st


def _check_rows(x, eps, rows, qsel=None):
    n = len(x)
    qsel = np.arange(n) if qsel is None else np.asarray(qsel)
    want = oracle.row_sets(x, eps, qsel)
    for k, q in enumerate(qsel.tolist()):
        sure, band = want[k]
        got = rows[q]
        g = set(got.tolist())
        assert len(g) == got.size, "duplicate neighbour in row %d" % q
        assert q in g
        assert sure <= g, "row %d misses %s" % (q, sorted(sure - g)[:5])
        assert g <= sure | band, "row %d has extra %s" % (q, sorted(g - sure - band)[:5])


def test_config1_full_pair_for_pair():
    x = datagen.generate(1)
    eps = golden_eps(1)
    rows, counts, st = _join(x, eps)
    assert len(rows) == len(x)
    _check_rows(x, eps, rows)
    true = oracle.counts(x, eps)
    assert np.all(counts >= true)
    assert st["pairs"] == sum(r.size for r in rows.values())


@pytest.mark.parametrize("cfg,n,k", [(1, 5000, 32), (2, 6000, 64), (3, 6000, 128), (4, 3000, 64), (5, 8000, 100)])
def test_small_workloads(cfg, n, k):
    x = datagen.generate(cfg, n=n)
    eps = oracle.pick_eps(x, k, datagen.sample_queries(n, 200, seed=cfg))["eps"]
    rows, counts, st = _join(x, eps)
    _check_rows(x, eps, rows)
    assert np.array_equal(counts, oracle.count_bound(x, eps))
    # every result pair lies in a staged tile the refinement kept
    assert st["pairs"] <= st["candidates_refined"] <= st["candidates"]


def test_stage_skip_keeps_every_neighbour():
    """Points spread along one axis (the other dimensions nearly constant):
    a 128-query tile covers part of its cell, so the 32-row groups at the far
    ends of the neighbouring cells are more than eps from it and their tiles
    are skipped before streaming.  The result must not change, and the
    tensor-core refinement (which streams every tile) reports -1."""
    rng = np.random.default_rng(5)
    n, d = 4096, 16
    x = rng.normal(0.0, 0.01, (n, d)).astype(np.float32)
    x[:, 0] = rng.uniform(0.0, 10.0, n).astype(np.float32)
    eps = 1.0
    rows, counts, st = _join(x, eps)
    _check_rows(x, eps, rows)
    assert st["pairs"] <= st["candidates_refined"] < st["candidates"]
    edd = _edd()
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    j.set_refine(True)
    rows_tc = j.join_sets(eps, 0)
    assert j.stats()["candidates_refined"] == -1
    j.close()
    _check_rows(x, eps, rows_tc)


@pytest.mark.parametrize("d", [1, 2, 3, 5, 17, 64, 127, 128, 130, 200, 256])
def test_dimensions(d):
    rng = np.random.default_rng(40 + d)
    n = 1500
    x = (rng.standard_normal((n, d)) * (np.arange(1, d + 1) ** -0.3)).astype(np.float32)
    eps = oracle.pick_eps(x, 20, np.arange(0, n, 10))["eps"]
    rows, counts, _ = _join(x, eps)
    _check_rows(x, eps, rows)
    assert np.array_equal(counts, oracle.count_bound(x, eps))


def test_eps_zero_duplicates_and_single_point():
    x = datagen.generate(1, n=500)
    x[100:110] = x[7]
    rows, counts, _ = _join(x, 0.0)
    for q in range(len(x)):
        want = {q} if not (q == 7 or 100 <= q < 110) else {7, *range(100, 110)}
        assert set(rows[q].tolist()) == want
    rows, counts, _ = _join(x[:1], 1.0)
    assert rows[0].tolist() == [0] and counts.tolist() == [1]


@pytest.mark.parametrize("d", [3, 16, 32, 64, 128])
@pytest.mark.parametrize("eps", [2.0, 3.0])
def test_exact_boundary_on_integer_lattice(d, eps):
    """Integer coordinates make every float32 operation of the refinement
    exact, so the rows must equal the definition with no tolerance band:
    pairs at exactly eps are in, pairs beyond are out.  Many pairs lie
    exactly on the boundary, among them pairs whose query and candidate
    boxes over the three index dimensions are exactly eps apart, which the
    warp-tile box test must not skip (d <= 32), and pairs that the survivor
    mode finishes one per lane (d = 64, 128)."""
    x = datagen.lattice(4000, d, seed=d, p_low=min(0.1, 1.2 / max(d - 3, 1)))
    rows, counts, _ = _join(x, eps)
    row_ptr, cols, _, dist2 = oracle.rows(x, eps, np.arange(len(x)), band=0.0)
    assert np.any(dist2 == eps * eps), "no pair exactly on the boundary"
    for q in range(len(x)):
        want = cols[row_ptr[q]:row_ptr[q + 1]]
        assert np.array_equal(np.sort(rows[q]), want), "row %d differs" % q
        assert counts[q] >= want.size


def test_eps_covering_everything_and_tiny_eps():
    x = datagen.generate(1, n=1200)
    rows, counts, _ = _join(x, 10.0)
    assert all(r.size == len(x) for r in rows.values())
    assert np.all(counts == len(x))
    rows, counts, st = _join(x, 1e-4)
    assert all(r.tolist() == [q] for q, r in rows.items())
    assert st["cells"] > 1


def test_index_matches_oracle_grid():
    edd = _edd()
    x = datagen.generate(2, n=5000)
    eps = 6.0
    g = oracle.grid(x, eps)
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    j.count(eps)
    ix = j.index()
    assert ix["perm"] == g["perm"][:3].tolist()
    assert ix["cell_width"] == g["w"] and ix["sub_bits"] == g["sub_bits"]
    assert np.array_equal(ix["ids"].cpu().numpy(), g["order"])
    assert np.array_equal(ix["cell_start"].cpu().numpy(), g["cell_start"])
    assert np.array_equal(ix["cell_key"].cpu().numpy().view(np.uint64), g["cell_key"])
    st = oracle.stencil(g)
    nbr = ix["nbr"].cpu().numpy().reshape(-1, 27)
    cnt = ix["nbr_count"].cpu().numpy()
    for c in range(ix["cells"]):
        assert nbr[c, :cnt[c]].tolist() == st[c]
    j.close()


def test_mask_mode_bits():
    edd = _edd()
    x = datagen.generate(1, n=3000)
    eps = 0.55
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    j.count(eps)
    ix = j.index()
    ids = ix["ids"].cpu().numpy()
    cs = ix["cell_start"].cpu().numpy()
    nbr = ix["nbr"].cpu().numpy().reshape(-1, 27)
    cnt = ix["nbr_count"].cpu().numpy()
    cor = ix["cell_of_row"].cpu().numpy()
    got = {}

    def take(b):
        rp = edd._host_array(b.row_ptr, b.nq + 1, np.int64)
        words = edd._host_array(b.mask, b.n_words, np.uint32)
        cand = edd._host_array(b.cand, b.nq, np.int64)
        qrows = edd._host_array(b.query_rows, b.nq, np.int32)
        qids = edd._host_array(b.query_ids, b.nq, np.int64)
        for i in range(b.nq):
            bits = np.unpackbits(words[rp[i]:rp[i + 1]].view(np.uint8), bitorder="little")[:cand[i]]
            c = cor[qrows[i]]
            members = np.concatenate([ids[cs[nb]:cs[nb + 1]] for nb in nbr[c, :cnt[c]]])
            assert members.size == cand[i]
            got[int(qids[i])] = members[bits.astype(bool)]

    j.join(eps, 0, edd.HISS_OUT_MASK, True, take)
    j.close()
    _check_rows(x, eps, got)


def test_batching_matches_single_batch():
    x = datagen.generate(5, n=20000)
    eps = 0.7
    rows1, _, st1 = _join(x, eps)
    rows2, _, st2 = _join(x, eps, batch_bytes=1 << 20)
    assert st1["batches"] == 1 and st2["batches"] > 5
    for q in range(len(x)):
        assert np.array_equal(np.sort(rows1[q]), np.sort(rows2[q]))
    _check_rows(x, eps, rows2, np.arange(0, len(x), 37))


@pytest.mark.parametrize("copy_to_host", [False, True])
def test_dense_result_comes_in_parts_within_batch_bytes(copy_to_host):
    # eps covers every pair, so the CSR result (n^2 ids, 64 MB) is 32 times
    # the result mask (2 MB).  With batch_bytes = 8 MB the mask fits in one
    # batch but its CSR does not: the join must hand the batch over in parts
    # that fit, and the context must stay under an allocation cap that the
    # whole CSR would break, instead of failing with HISS_E_NOMEM.
    edd = _edd()
    x = datagen.generate(1, n=4000)          # U[0,1)^16: every distance < 4
    n, eps = len(x), 10.0
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    j.set_alloc_limit(40 << 20)
    rows, nq_seen, idx = {}, [0], []

    def take(b):
        idx.append(int(b.index))
        if copy_to_host:
            q = edd._host_array(b.query_ids, b.nq, np.int64)
            rp = edd._host_array(b.row_ptr, b.nq + 1, np.int64)
            cols = edd._host_array(b.cols, b.nnz, np.int32)
        else:
            q = torch.as_tensor(edd.DeviceArray(b.query_ids, (b.nq,), "<i8"), device="cuda").cpu().numpy()
            rp = torch.as_tensor(edd.DeviceArray(b.row_ptr, (b.nq + 1,), "<i8"), device="cuda").cpu().numpy()
            cols = torch.as_tensor(edd.DeviceArray(b.cols, (b.nnz,), "<i4"), device="cuda").cpu().numpy()
        assert rp[0] == 0 and rp[-1] == b.nnz and 4 * b.nnz <= 8 << 20
        nq_seen[0] += b.nq
        for i in range(b.nq):
            assert int(q[i]) not in rows
            rows[int(q[i])] = np.sort(cols[rp[i]:rp[i + 1]])

    st = j.join(eps, 8 << 20, edd.HISS_OUT_CSR, copy_to_host, take)
    j.close()
    assert st["pairs"] == n * n
    assert st["deliveries"] > st["batches"] >= 1
    assert idx == list(range(st["deliveries"]))
    assert nq_seen[0] == n and sorted(rows) == list(range(n))
    everyone = np.arange(n)
    for q in range(n):
        assert np.array_equal(rows[q], everyone)


def test_device_and_host_delivery_agree():
    edd = _edd()
    x = datagen.generate(3, n=4000)
    eps = 0.3
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    dev = {}

    def take(b):
        q = torch.as_tensor(edd.DeviceArray(b.query_ids, (b.nq,), "<i8"), device="cuda").cpu().numpy()
        rp = torch.as_tensor(edd.DeviceArray(b.row_ptr, (b.nq + 1,), "<i8"), device="cuda").cpu().numpy()
        cols = torch.as_tensor(edd.DeviceArray(b.cols, (max(b.nnz, 1),), "<i4"), device="cuda").cpu().numpy()
        for i in range(b.nq):
            dev[int(q[i])] = np.sort(cols[rp[i]:rp[i + 1]])

    j.join(eps, 0, edd.HISS_OUT_CSR, False, take)
    host = j.join_sets(eps)
    j.close()
    for q in range(len(x)):
        assert np.array_equal(dev[q], np.sort(host[q]))


def test_overlapped_host_delivery_many_batches_and_callback_stop():
    # CSR to host with many batches: copies of batch b overlap the refinement
    # of batch b + 1 (two pinned slots); the rows must match device delivery,
    # batches arrive in order, and a callback that stops the join leaves the
    # context usable
    edd = _edd()
    x = datagen.generate(2, n=8000)
    eps = oracle.pick_eps(x, 40, np.arange(0, 8000, 20))["eps"]
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    host, order = {}, []

    def take(b):
        order.append(int(b.index))
        q = edd._host_array(b.query_ids, b.nq, np.int64)
        rp = edd._host_array(b.row_ptr, b.nq + 1, np.int64)
        cols = edd._host_array(b.cols, b.nnz, np.int32)
        assert b.on_host == 1
        for i in range(b.nq):
            host[int(q[i])] = np.sort(cols[rp[i]:rp[i + 1]])

    st = j.join(eps, 1 << 16, edd.HISS_OUT_CSR, True, take)
    assert st["batches"] >= 3 and order == list(range(st["deliveries"]))
    dev = j.join_sets(eps)  # one batch
    assert set(host) == set(dev) == set(range(len(x)))
    for q in range(len(x)):
        assert np.array_equal(host[q], np.sort(dev[q]))
    calls = [0]

    def stop(b):
        calls[0] += 1
        if calls[0] == 2:
            raise RuntimeError("stop")

    with pytest.raises(RuntimeError):
        j.join(eps, 1 << 16, edd.HISS_OUT_CSR, True, stop)
    again = j.join_sets(eps, 1 << 16)
    assert all(np.array_equal(np.sort(again[q]), np.sort(dev[q])) for q in range(len(x)))
    j.close()


def test_refine_option_values():
    edd = _edd()
    import ctypes
    j = edd.Join()
    for v in (2, -1, 7):
        assert edd.hiss_set_option(j.handle, edd.HISS_OPT_REFINE, v) == edd.HISS_E_ARG
    assert edd.hiss_set_option(j.handle, 99, 0) == edd.HISS_E_ARG
    j.close()


def test_host_build_matches_device_build():
    edd = _edd()
    x = datagen.generate(4, n=2000)
    eps = 1.2
    j = edd.Join()
    j.build(x)
    a = j.join_sets(eps)
    j.build(torch.from_numpy(x).cuda())
    b = j.join_sets(eps)
    j.close()
    for q in range(len(x)):
        assert np.array_equal(np.sort(a[q]), np.sort(b[q]))


def test_error_statuses():
    edd = _edd()
    j = edd.Join()
    with pytest.raises(edd.HissError) as e:
        j.join(1.0)
    assert e.value.status == edd.HISS_E_STATE
    x = datagen.generate(1, n=100)
    bad = x.copy()
    bad[5, 3] = np.nan
    with pytest.raises(edd.HissError) as e:
        j.build(torch.from_numpy(bad).cuda())
    assert e.value.status == edd.HISS_E_ARG
    j.build(torch.from_numpy(x).cuda())
    for eps in (-1.0, float("nan"), float("inf")):
        with pytest.raises(edd.HissError) as e:
            j.join(eps)
        assert e.value.status == edd.HISS_E_ARG
    with pytest.raises(edd.HissError) as e:
        j.join(0.5, batch_bytes=16)
    assert e.value.status == edd.HISS_E_BATCH_TOO_SMALL

    def stop(b):
        raise KeyError("stop")

    with pytest.raises(KeyError):
        j.join(0.5, on_batch=stop)
    # the context stays usable after host-side errors
    assert len(j.join_sets(0.5)) == 100
    j.close()
    with pytest.raises(edd.HissError) as e:
        j2 = edd.Join()
        j2.set_alloc_limit(1 << 12)
        j2.build(torch.from_numpy(x).cuda())
    assert e.value.status == edd.HISS_E_NOMEM
    rc = edd.hiss_build(None, None, 10, 3)
    assert rc == edd.HISS_E_ARG


def _exit_dims_reference(xs, eps, cell_start, nbr, nbr_count, cell_of_row, d):
    """Sum over candidate pairs of the dimensions needed when a pair stops at
    the first multiple of 4 whose float32 partial sum exceeds eps^2 (the
    kernel's own arithmetic: a float32 product, then fused multiply-adds)."""
    e2 = np.float32(eps) * np.float32(eps)
    total = 0
    for q in range(xs.shape[0]):
        c = cell_of_row[q]
        cand = np.concatenate([np.arange(cell_start[nb], cell_start[nb + 1]) for nb in nbr[c, :nbr_count[c]]])
        e = (xs[q][None, :] - xs[cand]).astype(np.float32)
        acc = (e[:, 0] * e[:, 0]).astype(np.float32)
        alive = np.ones(cand.size, bool)
        dims = np.zeros(cand.size, np.int64)
        for k in range(1, xs.shape[1]):
            acc = (acc.astype(np.float64) + e[:, k].astype(np.float64) ** 2).astype(np.float32)
            if (k + 1) % 4 == 0 or k + 1 == xs.shape[1]:
                step_end = min(k + 1, d)
                dims[alive] = step_end
                alive &= acc <= e2
        total += int(dims.sum())
    return total


def test_work_profile_counts_early_exit_dimensions():
    edd = _edd()
    x = datagen.generate(2, n=3000)
    eps = 6.0
    j = edd.Join()
    j.build(torch.from_numpy(x).cuda())
    j.count(eps)
    st = j.stats()
    alg, executed = j.work_profile(eps)
    ix = j.index()
    g = oracle.grid(x, eps)
    perm = oracle.variance_order(oracle.dim_stats(x)[2])
    d = x.shape[1]
    xs = x[:, perm][g["order"]]
    want = _exit_dims_reference(xs, eps, ix["cell_start"].cpu().numpy(),
                                ix["nbr"].cpu().numpy().reshape(-1, 27), ix["nbr_count"].cpu().numpy(),
                                ix["cell_of_row"].cpu().numpy(), d)
    j.close()
    assert abs(alg - want) <= 1e-6 * want + 8, (alg, want)
    # a warp skips a block of pairs whose boxes over the three index
    # dimensions are farther apart than eps, and otherwise checks every 2
    # dimensions (d4 <= 64): at most d4 per pair
    assert 0 < executed <= st["candidates"] * (d + 8)
