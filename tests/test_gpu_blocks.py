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
