"""Seeded synthetic point sets for the exact epsilon self-join.

This module only draws random numbers: it holds none of the join's
arithmetic (no distances, no grid, no selection), so both the CPU oracle
tests and the CUDA path tests can draw their inputs from it.

The five workloads stand in for the real-world datasets of RT-HiSS
(Munugala & Gowanlock, "RT-HiSS: Ray Tracing Accelerated High Dimensional
Vector Similarity Searches", Table I), which are not available here:

  1. uniform    N=20,000   d=16   i.i.d. U[0,1)
  2. gmm        N=1,000,000 d=32  200-centre Gaussian mixture, centres
                U[0,100)^d, per-cluster sigma U[0.5,3], cluster sizes with
                Zipf(1.1) shares
  3. subspace   N=2,000,000 d=64  random 8-dim linear subspace, Gaussian
                coefficients sigma=1, plus isotropic noise sigma=0.01
  4. spectrum   N=500,000  d=128  N(0,1) coordinates scaled by k^-0.7
  5. exp        N=5,000,000 d=16  i.i.d. exponential(lambda=1)

Every value is drawn in float64 by NumPy's PCG64 and then cast to float32;
the float32 array is the dataset of record.  ``n`` may be given to draw a
smaller instance of the same distribution (for parity tests); the stream is
then a different one, seeded by (master, config, n).
"""
from __future__ import annotations

import numpy as np

MASTER_SEED = 20260902

# (name, N, d, target mean neighbours per point, self excluded)
CONFIGS = {
    1: ("uniform", 20_000, 16, 32),
    2: ("gmm", 1_000_000, 32, 64),
    3: ("subspace", 2_000_000, 64, 128),
    4: ("spectrum", 500_000, 128, 256),
    5: ("exp", 5_000_000, 16, 1000),
}


def _rng(cfg: int, n: int | None) -> np.random.Generator:
    key = [MASTER_SEED, cfg] if n is None else [MASTER_SEED, cfg, int(n)]
    return np.random.default_rng(key)


def _zipf_sizes(n: int, n_clusters: int, s: float, rng: np.random.Generator) -> np.ndarray:
    """Cluster sizes with shares proportional to r^-s (r = 1..n_clusters),
    rounded to integers summing to n by the largest-remainder rule, then
    assigned to the centres by a seeded permutation."""
    r = np.arange(1, n_clusters + 1, dtype=np.float64)
    share = r ** (-s)
    share /= share.sum()
    exact = share * n
    base = np.floor(exact).astype(np.int64)
    rem = n - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:rem]] += 1
    return base[rng.permutation(n_clusters)]


def generate(cfg: int, n: int | None = None) -> np.ndarray:
    """Return the float32 (N, d) row-major point set of workload ``cfg``."""
    name, n_full, d, _ = CONFIGS[cfg]
    n = n_full if n is None else int(n)
    rng = _rng(cfg, None if n == n_full else n)
    if name == "uniform":
        x = rng.random((n, d))
    elif name == "gmm":
        k = 200
        centres = rng.random((k, d)) * 100.0
        sigma = rng.uniform(0.5, 3.0, size=k)
        sizes = _zipf_sizes(n, k, 1.1, rng)
        label = np.repeat(np.arange(k), sizes)
        x = centres[label] + sigma[label, None] * rng.standard_normal((n, d))
        x = x[rng.permutation(n)]
    elif name == "subspace":
        basis, _ = np.linalg.qr(rng.standard_normal((d, 8)))
        coef = rng.standard_normal((n, 8))
        x = coef @ basis.T + 0.01 * rng.standard_normal((n, d))
    elif name == "spectrum":
        scale = np.arange(1, d + 1, dtype=np.float64) ** (-0.7)
        x = rng.standard_normal((n, d)) * scale
    elif name == "exp":
        x = rng.exponential(1.0, size=(n, d))
    else:  # pragma: no cover
        raise ValueError(name)
    return np.ascontiguousarray(x.astype(np.float32))


def lattice(n: int, d: int, seed: int, side: int = 20, p_low: float = 0.1) -> np.ndarray:
    """Integer points for exact-boundary tests: the first min(d, 3)
    coordinates uniform on {0, ..., side - 1}, the others 1 with probability
    p_low and 0 otherwise (so the first three have the largest variance).
    Every squared distance is a small integer, exact in float32."""
    rng = np.random.default_rng([MASTER_SEED, 99, int(n), int(d), int(seed)])
    x = np.zeros((n, d), dtype=np.float64)
    k = min(d, 3)
    x[:, :k] = rng.integers(0, side, size=(n, k))
    if d > k:
        x[:, k:] = (rng.random((n, d - k)) < p_low).astype(np.float64)
    return np.ascontiguousarray(x.astype(np.float32))


def sample_queries(n: int, m: int, seed: int) -> np.ndarray:
    """m distinct query indices in [0, n), drawn without replacement."""
    return np.random.default_rng(seed).choice(n, size=min(m, n), replace=False).astype(np.int64)


def describe(cfg: int) -> dict:
    name, n, d, k = CONFIGS[cfg]
    return {"workload": name, "n": n, "d": d, "mean_neighbours": k}
