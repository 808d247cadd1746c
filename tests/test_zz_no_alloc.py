"""hiss_exclusive_scan_noalloc: the exclusive scan for callers that cannot
allocate device memory (a plugin whose host framework owns all device memory,
or a loop that cannot afford cudaMalloc's implicit synchronisation).  It keeps
its scratch in a static device array instead of context buffers.

Checked through the C ABI against a host prefix sum (numpy) and against
hiss_exclusive_scan, on consecutive calls that share the static scratch:
ragged sizes, n = 0, the documented in-place call (input and output the same
buffer), and n at the 2^26 limit, where the scratch is fullest."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _host_exclusive(x):
    out = np.zeros(x.size + 1, dtype=np.int64)
    np.cumsum(x, out=out[1:])
    return out


def test_noalloc_scan_matches_host_and_context_scan():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    h = ctypes.c_void_p()
    assert edd.hiss_create(ctypes.byref(h), sp) == edd.HISS_OK
    try:
        # two calls in a row at each size: the second sees the scratch the first left
        for call, n in enumerate([1_000_003, 4097, 1, 2048, 2049, 1 << 26]):
            rng = np.random.default_rng(100 + call)
            xh = rng.integers(-(1 << 30), 1 << 30, size=n, dtype=np.int64)
            want_h = _host_exclusive(xh)
            x = torch.from_numpy(xh).cuda()
            want = torch.empty(n + 1, dtype=torch.int64, device="cuda")
            assert edd.hiss_exclusive_scan(h, x.data_ptr(), want.data_ptr(), n) == edd.HISS_OK
            for rep in range(2):
                got = torch.full((n + 1,), -7, dtype=torch.int64, device="cuda")
                assert edd.hiss_exclusive_scan_noalloc(sp, x.data_ptr(), got.data_ptr(), n) == edd.HISS_OK
                torch.cuda.synchronize()
                assert np.array_equal(got.cpu().numpy(), want_h), "n=%d call %d differs from numpy" % (n, rep)
                assert torch.equal(got, want), "n=%d call %d differs from hiss_exclusive_scan" % (n, rep)
            del x, want, got
        # in place: input and output are the same buffer (n + 1 entries)
        n = 300_001
        xh = np.random.default_rng(7).integers(0, 1 << 20, size=n, dtype=np.int64)
        buf = torch.zeros(n + 1, dtype=torch.int64, device="cuda")
        buf[:n] = torch.from_numpy(xh).cuda()
        assert edd.hiss_exclusive_scan_noalloc(sp, buf.data_ptr(), buf.data_ptr(), n) == edd.HISS_OK
        torch.cuda.synchronize()
        assert np.array_equal(buf.cpu().numpy(), _host_exclusive(xh))
        # n = 0: out[0] = 0, the input is not read
        z = torch.full((1,), 99, dtype=torch.int64, device="cuda")
        assert edd.hiss_exclusive_scan_noalloc(sp, None, z.data_ptr(), 0) == edd.HISS_OK
        torch.cuda.synchronize()
        assert int(z.item()) == 0
        # beyond the limit: rejected before any launch
        too_big = (1 << 26) + 1
        assert edd.hiss_exclusive_scan_noalloc(sp, buf.data_ptr(), buf.data_ptr(), too_big) == edd.HISS_E_ARG
        assert edd.hiss_exclusive_scan_noalloc(sp, buf.data_ptr(), None, 5) == edd.HISS_E_ARG
    finally:
        edd.hiss_destroy(h)
