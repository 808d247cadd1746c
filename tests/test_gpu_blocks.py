"""The building blocks of the join on the GPU, through the C ABI: the onesweep
radix sort (against a stable sort), the exclusive scan, and the result-mask
compaction of Fig. 5."""
import numpy as np
import pytest

import oracle
from conftest import read_golden

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd
    j = edd.Join()
    yield j
    j.close()


@pytest.mark.parametrize("n", [2, 31, 4095, 4096, 4097, 100_003, (1 << 20) + 7])
@pytest.mark.parametrize("bits", [1, 7, 8, 13, 32, 63, 64])
def test_sort_is_stable_lsd(ctx, n, bits):
    rng = np.random.default_rng(n * 131 + bits)
    keys = rng.integers(0, 1 << 63, size=n, dtype=np.int64).view(np.uint64) * np.uint64(2) + \
        rng.integers(0, 2, size=n).astype(np.uint64)
    if bits < 64:
        keys_masked = keys & np.uint64((1 << bits) - 1)
    else:
        keys_masked = keys
    if n > 1000:
        keys[: n // 3] = keys[n // 2]  # long runs of equal keys
        keys_masked = keys & np.uint64((1 << bits) - 1) if bits < 64 else keys
    vals = np.arange(n, dtype=np.uint32)
    kt = torch.from_numpy(keys.view(np.int64).copy()).cuda()
    vt = torch.from_numpy(vals.view(np.int32).copy()).cuda()
    ctx.sort_pairs(kt, vt, bits)
    order = np.argsort(keys_masked, kind="stable")
    assert np.array_equal(vt.cpu().numpy().view(np.uint32), order.astype(np.uint32))
    assert np.array_equal(kt.cpu().numpy().view(np.uint64), keys[order])


@pytest.mark.parametrize("n", [0, 1, 2047, 2048, 2049, 1_000_001])
def test_exclusive_scan(ctx, n):
    rng = np.random.default_rng(n)
    x = rng.integers(0, 1 << 20, size=n, dtype=np.int64)
    xt = torch.from_numpy(x).cuda()
    out = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    ctx.exclusive_scan(xt, out)
    want = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(x, out=want[1:])
    assert np.array_equal(out.cpu().numpy(), want)


def _pack(bits):
    b = np.zeros(((len(bits) + 31) // 32) * 32, dtype=np.uint8)
    b[: len(bits)] = bits
    return np.packbits(b, bitorder="little").view(np.uint32)


def test_fig5_compaction_on_gpu(ctx):
    g = dict(read_golden("fig5_mask.txt"))
    bits = np.array([int(v) for v in g["mask"]], dtype=np.uint8)
    words = torch.from_numpy(_pack(bits).view(np.int32).copy()).cuda()
    pos = torch.full((len(bits),), -1, dtype=torch.int64, device="cuda")
    cnt = ctx.mask_positions(words, len(bits), pos)
    assert pos[:cnt].cpu().tolist() == [int(v) for v in g["positions"]]


@pytest.mark.parametrize("nbits", [1, 31, 32, 33, 100_000])
def test_compaction_random_masks(ctx, nbits):
    rng = np.random.default_rng(nbits)
    bits = (rng.random(nbits) < 0.1).astype(np.uint8)
    words = _pack(bits)
    words_t = torch.from_numpy(words.view(np.int32).copy()).cuda()
    pos = torch.empty(nbits, dtype=torch.int64, device="cuda")
    cnt = ctx.mask_positions(words_t, nbits, pos)
    assert np.array_equal(pos[:cnt].cpu().numpy(), oracle.compact_mask(bits))


def _tf32_rna(x):
    """float32 -> TF32 (10 explicit mantissa bits), to nearest, ties away
    from zero, done on the bit pattern (test-side restatement of the
    rounding that the tensor-core operands get)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).astype(np.uint32)
    return r.view(np.float32)


@pytest.mark.parametrize("k", [8, 16, 40, 72, 128])
def test_gram_tf32_on_tensor_cores(ctx, k):
    import ctypes
    import exact_dimensional_distance_gb300 as edd
    rng = np.random.default_rng(500 + k)
    a = (rng.standard_normal((128, k)) * rng.uniform(0.1, 10, size=(128, 1))).astype(np.float32)
    b = (rng.standard_normal((128, k)) * rng.uniform(0.1, 10, size=(128, 1))).astype(np.float32)
    a[5, :] = 0.0          # an all-zero row
    b[:, 3] = 1.0          # a constant column
    at, bt = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda")
    rc = edd.hiss_gram_tf32(ctx._h, ctypes.c_void_p(at.data_ptr()), ctypes.c_void_p(bt.data_ptr()), k,
                            ctypes.c_void_p(out.data_ptr()))
    assert rc == edd.HISS_OK, edd.hiss_strerror(rc)
    ta, tb = _tf32_rna(a).astype(np.float64), _tf32_rna(b).astype(np.float64)
    want = ta @ tb.T
    # float32 accumulation of k exact products: error <= k 2^-22 sum |a_k b_k|
    bound = (k + 8) * 2.0 ** -22 * (np.abs(ta) @ np.abs(tb).T) + 1e-30
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) / bound))
    # TF32 rounding really happened (operands are not used at float32 precision)
    assert not np.allclose(ta, a.astype(np.float64), rtol=0, atol=0)
