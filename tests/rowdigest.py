"""Row fingerprints for comparing large join rows without listing them.

splitmix64 here is written independently of the oracle's C version (numpy
uint64 arithmetic, which wraps modulo 2^64); the tests check it against the
generator's published outputs.  A row's digest is (count, sum of
splitmix64(j) modulo 2^64 over its neighbour ids j)."""
import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(v) -> np.ndarray:
    """First output of a splitmix64 generator seeded with each v."""
    with np.errstate(over="ignore"):
        z = np.asarray(v, dtype=np.uint64) + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def row_hash(cols) -> int:
    """Sum modulo 2^64 of splitmix64 over a row's neighbour ids."""
    cols = np.asarray(cols)
    if cols.size == 0:
        return 0
    with np.errstate(over="ignore"):
        return int(np.sum(splitmix64(cols.astype(np.uint64)), dtype=np.uint64))
