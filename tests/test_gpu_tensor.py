"""The tensor-core refinement (HISS_OPT_REFINE = HISS_REFINE_TENSOR_CORES)
against the fp64 oracle, through the C ABI: TF32 Gram-matrix estimates on
the tensor cores decide pairs outside a rigorous error margin, pairs inside
it are rechecked exactly, so the pair sets must equal the oracle's outside
the eps^2 band (and agree with the CUDA-core refinement there)."""
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


def _join(x, eps, batch_bytes=0, tensor=True):
    edd = _edd()
    j = edd.Join()
    j.set_refine(tensor)
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
        assert sure <= g, "row %d misses %s" % (q, sorted(sure - g)[:5])
        assert g <= sure | band, "row %d has extra %s" % (q, sorted(g - sure - band)[:5])


def test_config1_full_pair_for_pair_tensor():
    x = datagen.generate(1)
    eps = golden_eps(1)
    rows, counts, st = _join(x, eps)
    assert len(rows) == len(x)
    _check_rows(x, eps, rows)
    assert st["pairs"] == sum(r.size for r in rows.values())


@pytest.mark.parametrize("cfg,n,k", [(2, 6000, 64), (3, 6000, 128), (4, 3000, 64), (5, 8000, 100)])
def test_small_workloads_tensor(cfg, n, k):
    x = datagen.generate(cfg, n=n)
    eps = oracle.pick_eps(x, k, np.arange(0, n, max(1, n // 500)))["eps"]
    rows, counts, st = _join(x, eps)
    _check_rows(x, eps, rows)


@pytest.mark.parametrize("d", [1, 3, 5, 17, 64, 100, 128, 130])
def test_dimensions_tensor(d):
    rng = np.random.default_rng(70 + d)
    n = 1500
    x = (rng.standard_normal((n, d)) * (np.arange(1, d + 1) ** -0.3)).astype(np.float32)
    eps = oracle.pick_eps(x, 20, np.arange(0, n, 10))["eps"]
    rows, counts, st = _join(x, eps)
    _check_rows(x, eps, rows)


def test_tensor_and_cuda_cores_agree_outside_band():
    x = datagen.generate(2, n=5000)
    eps = oracle.pick_eps(x, 64, np.arange(0, 5000, 10))["eps"]
    a, _, sa = _join(x, eps, tensor=True)
    b, _, sb = _join(x, eps, tensor=False)
    want = oracle.row_sets(x, eps, np.arange(len(x)))
    for q in range(len(x)):
        sure, band = want[q]
        ga, gb = set(a[q].tolist()), set(b[q].tolist())
        assert ga - band == gb - band == sure


def test_far_offsets_and_exact_boundaries_tensor():
    # large common offset with a small eps: the margins are wide relative to
    # eps^2 unless the centring works; integer points give distances exactly
    # equal to eps (3-4-5 triangles), decided by the exact recheck
    rng = np.random.default_rng(9)
    base = rng.integers(0, 6, size=(800, 8)).astype(np.float32)
    x = np.concatenate([base + np.float32(4096.0), base * np.float32(0.5) - np.float32(1e4)]).astype(np.float32)
    for eps in (1.0, 5.0, 2.0 ** 0.5):
        rows, counts, st = _join(x, eps)
        _check_rows(x, eps, rows)


def test_many_batches_and_duplicates_tensor():
    x = datagen.generate(1, n=4000)
    x[100:140] = x[7]
    eps = golden_eps(1)
    rows, counts, st = _join(x, eps, batch_bytes=1 << 17)
    assert st["batches"] > 1
    _check_rows(x, eps, rows)
    rows0, _, _ = _join(x, 0.0)
    for q in range(len(x)):
        want = {q} if not (q == 7 or 100 <= q < 140) else {7, *range(100, 140)}
        assert set(rows0[q].tolist()) == want


def test_semi_join_tensor():
    edd = _edd()
    x = datagen.generate(2, n=4000)
    rng = np.random.default_rng(3)
    qx = (x[rng.choice(4000, 700, replace=False)] + rng.normal(0, 0.5, (700, x.shape[1]))).astype(np.float32)
    eps = oracle.pick_eps(x, 32, np.arange(0, 4000, 10))["eps"]
    j = edd.Join()
    j.set_refine(True)
    j.build(torch.from_numpy(x).cuda())
    got = j.join_queries_sets(torch.from_numpy(qx).cuda(), eps)
    j.close()
    want = oracle.semi_row_sets(qx, x, eps)
    for q in range(len(qx)):
        sure, band = want[q]
        g = set(got[q].tolist())
        assert sure <= g <= sure | band
