"""hiss_exclusive_scan_noalloc: the exclusive scan for callers that cannot
allocate device memory (a plugin whose host framework owns all device memory,
or a loop that cannot afford cudaMalloc's implicit synchronisation).  It keeps
its scratch in a static device array instead of context buffers.  Checked
through the C ABI against hiss_exclusive_scan on two calls in a row (the
second call sees the scratch the first one left behind)."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_noalloc_scan_matches_context_scan():
    import __graft_entry__
    __graft_entry__.build()
    import exact_dimensional_distance_gb300 as edd

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    h = ctypes.c_void_p()
    assert edd.hiss_create(ctypes.byref(h), ctypes.c_void_p(stream.cuda_stream)) == edd.HISS_OK
    try:
        for call, n in enumerate([1_000_003, 4097]):
            rng = np.random.default_rng(100 + call)
            x = torch.from_numpy(rng.integers(-(1 << 30), 1 << 30, size=n, dtype=np.int64)).cuda()
            want = torch.empty(n + 1, dtype=torch.int64, device="cuda")
            got = torch.full((n + 1,), -7, dtype=torch.int64, device="cuda")
            assert edd.hiss_exclusive_scan(h, x.data_ptr(), want.data_ptr(), n) == edd.HISS_OK
            rc = edd.hiss_exclusive_scan_noalloc(ctypes.c_void_p(stream.cuda_stream), x.data_ptr(),
                                                 got.data_ptr(), n)
            assert rc == edd.HISS_OK
            torch.cuda.synchronize()
            assert torch.equal(got, want), "call %d differs" % call
        too_big = (1 << 26) + 1
        assert edd.hiss_exclusive_scan_noalloc(ctypes.c_void_p(stream.cuda_stream), x.data_ptr(),
                                               got.data_ptr(), too_big) == edd.HISS_E_ARG
    finally:
        edd.hiss_destroy(h)
