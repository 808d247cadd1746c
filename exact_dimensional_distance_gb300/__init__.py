"""GB300 exact epsilon self-join: thin Python binding of libhiss.so.

The library (include/hiss.h) computes the Euclidean self-join of RT-HiSS
(Munugala & Gowanlock, "RT-HiSS: Ray Tracing Accelerated High Dimensional
Vector Similarity Searches", Section II-A): every pair of points within eps,
self pairs included.  This module only marshals arguments: every step of the
join runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no CPU fallback: importing this module fails if
libhiss.so has not been built (``python exact_dimensional_distance_gb300/build.py``).

Functions with the names of the C ABI (``hiss_create``, ``hiss_build``, ...)
are the raw entry points; ``Join`` wraps a context for convenience.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhiss.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libhiss.so is missing: build it with "
                      "`python exact_dimensional_distance_gb300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

HISS_OK = 0
HISS_E_ARG = -1
HISS_E_NOMEM = -2
HISS_E_STATE = -3
HISS_E_BATCH_TOO_SMALL = -4
HISS_E_OVERFLOW = -5
HISS_E_CUDA = -6
HISS_E_CALLBACK = -7
HISS_OUT_CSR = 0
HISS_OUT_MASK = 1
HISS_OPT_ALLOC_LIMIT = 1
HISS_OPT_REFINE = 2
HISS_REFINE_CUDA_CORES = 0
HISS_REFINE_TENSOR_CORES = 1
HISS_MAX_DIM = 256

_i64, _i32, _f32, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class hiss_batch(ctypes.Structure):
    _fields_ = [("index", _i64), ("nq", _i64), ("query_ids", _p), ("row_ptr", _p), ("cols", _p),
                ("mask", _p), ("cand", _p), ("query_rows", _p), ("nnz", _i64), ("n_words", _i64),
                ("on_host", _i32), ("mode", _i32)]


HISS_BATCH_FN = ctypes.CFUNCTYPE(ctypes.c_int, _p, ctypes.POINTER(hiss_batch))


class hiss_out(ctypes.Structure):
    _fields_ = [("mode", _i32), ("copy_to_host", _i32), ("on_batch", HISS_BATCH_FN), ("user", _p)]


class hiss_index_view(ctypes.Structure):
    _fields_ = [("n", _i64), ("cells", _i64), ("ids", _p), ("cell_start", _p), ("cell_of_row", _p),
                ("nbr", _p), ("nbr_count", _p), ("cell_bound", _p), ("cell_key", _p),
                ("perm", _i32 * 3), ("sub_bits", _i32), ("cell_width", ctypes.c_double),
                ("origin", ctypes.c_double * 3)]


class hiss_stats(ctypes.Structure):
    _fields_ = [("n", _i64), ("cells", _i64), ("cell_pairs", _i64), ("candidates", _i64), ("pairs", _i64),
                ("batches", _i64), ("query_tiles", _i64), ("refine_units", _i64), ("mask_words_max", _i64),
                ("kernel_launches", _i64), ("d", _i32), ("d_pad", _i32), ("sub_bits", _i32),
                ("key_bits", _i32), ("eps", _f32), ("cell_width", ctypes.c_double),
                ("ms_build", ctypes.c_double), ("ms_index", ctypes.c_double), ("ms_count", ctypes.c_double),
                ("ms_refine", ctypes.c_double), ("ms_compact", ctypes.c_double),
                ("ms_deliver", ctypes.c_double), ("ms_total", ctypes.c_double), ("deliveries", _i64),
                ("candidates_refined", _i64)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


hiss_create = _sig("hiss_create", ctypes.c_int, [ctypes.POINTER(_p), _p])
hiss_destroy = _sig("hiss_destroy", None, [_p])
hiss_build = _sig("hiss_build", ctypes.c_int, [_p, _p, _i64, _i32])
hiss_build_host = _sig("hiss_build_host", ctypes.c_int, [_p, _p, _i64, _i32])
hiss_count = _sig("hiss_count", ctypes.c_int, [_p, _f32, _p])
hiss_join = _sig("hiss_join", ctypes.c_int, [_p, _f32, ctypes.c_size_t, ctypes.POINTER(hiss_out)])
hiss_index = _sig("hiss_index", ctypes.c_int, [_p, ctypes.POINTER(hiss_index_view)])
hiss_last_stats = _sig("hiss_last_stats", ctypes.c_int, [_p, ctypes.POINTER(hiss_stats)])
hiss_launch_count = _sig("hiss_launch_count", _i64, [_p])
hiss_strerror = _sig("hiss_strerror", ctypes.c_char_p, [ctypes.c_int])
hiss_last_cuda_error = _sig("hiss_last_cuda_error", ctypes.c_char_p, [_p])
hiss_set_option = _sig("hiss_set_option", ctypes.c_int, [_p, ctypes.c_int, _i64])
hiss_sort_pairs = _sig("hiss_sort_pairs", ctypes.c_int, [_p, _p, _p, _i64, _i32])
hiss_exclusive_scan = _sig("hiss_exclusive_scan", ctypes.c_int, [_p, _p, _p, _i64])
hiss_mask_positions = _sig("hiss_mask_positions", ctypes.c_int, [_p, _p, _i64, _p, ctypes.POINTER(_i64)])
hiss_work_profile = _sig("hiss_work_profile", ctypes.c_int, [_p, _f32, _p])
hiss_join_queries = _sig("hiss_join_queries", ctypes.c_int,
                         [_p, _p, _i64, _f32, ctypes.c_size_t, ctypes.POINTER(hiss_out)])
hiss_count_queries = _sig("hiss_count_queries", ctypes.c_int, [_p, _p, _i64, _f32, _p])
hiss_exclusive_scan_noalloc = _sig("hiss_exclusive_scan_noalloc", ctypes.c_int, [_p, _p, _p, _i64])
hiss_gram_tf32 = _sig("hiss_gram_tf32", ctypes.c_int, [_p, _p, _p, _i32, _p])
hiss_knn = _sig("hiss_knn", ctypes.c_int, [_p, _i32, _f32, _p, _p])
hiss_join_shard = _sig("hiss_join_shard", ctypes.c_int,
                       [_p, _f32, ctypes.c_size_t, ctypes.POINTER(hiss_out), _i32, _i32])

EXPORTED = ["hiss_create", "hiss_destroy", "hiss_build", "hiss_build_host", "hiss_count", "hiss_join",
            "hiss_index", "hiss_last_stats", "hiss_launch_count", "hiss_strerror", "hiss_last_cuda_error",
            "hiss_set_option", "hiss_sort_pairs", "hiss_exclusive_scan", "hiss_mask_positions",
            "hiss_exclusive_scan_noalloc", "hiss_work_profile", "hiss_join_queries", "hiss_count_queries",
            "hiss_gram_tf32", "hiss_knn", "hiss_join_shard"]


class HissError(RuntimeError):
    def __init__(self, status, ctx=None, what=""):
        msg = hiss_strerror(status).decode()
        if status == HISS_E_CUDA and ctx:
            msg += " (" + hiss_last_cuda_error(ctx).decode() + ")"
        super().__init__("%s: %s [%d]" % (what, msg, status))
        self.status = status


def _check(rc, ctx=None, what=""):
    if rc != HISS_OK:
        raise HissError(rc, ctx, what)


class DeviceArray:
    """A library-owned device buffer exposed through __cuda_array_interface__
    (wrap with torch.as_tensor(a, device='cuda'))."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr or 0), False), "version": 3}


def _host_array(ptr, n, dtype):
    if n == 0:
        return np.zeros(0, dtype=dtype)
    ctype = np.ctypeslib.as_ctypes_type(np.dtype(dtype))
    return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctype)), shape=(n,)).copy()


def _device_tensor(ptr, n, typestr):
    import torch
    if n == 0:
        return torch.zeros(0, dtype={"<i8": torch.int64, "<i4": torch.int32, "<u4": torch.int32}[typestr],
                           device="cuda")
    return torch.as_tensor(DeviceArray(ptr, (n,), typestr), device="cuda")


class Join:
    """One library context on a torch CUDA stream (default: the current one)."""

    def __init__(self, stream=None):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("a CUDA device is required")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = _p()
        _check(hiss_create(ctypes.byref(h), _p(self.stream.cuda_stream)), None, "hiss_create")
        self._h = h
        self.n = 0
        self.d = 0

    def close(self):
        if getattr(self, "_h", None):
            hiss_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def build(self, points):
        """points: torch CUDA float32 (n, d) tensor, or a numpy float32 (n, d) array."""
        if isinstance(points, np.ndarray):
            x = np.ascontiguousarray(points, dtype=np.float32)
            _check(hiss_build_host(self._h, x.ctypes.data, x.shape[0], x.shape[1]), self._h, "hiss_build_host")
            self.n, self.d = x.shape
            return self
        import torch
        assert points.is_cuda and points.dtype == torch.float32 and points.dim() == 2
        x = points.contiguous()
        _check(hiss_build(self._h, x.data_ptr(), x.shape[0], x.shape[1]), self._h, "hiss_build")
        self.n, self.d = x.shape
        return self

    def count(self, eps, out=None):
        """Count bound B_q of every point (int64 torch CUDA tensor, original order)."""
        import torch
        if out is None:
            out = torch.empty(self.n, dtype=torch.int64, device="cuda")
        _check(hiss_count(self._h, float(eps), out.data_ptr() if out is not False else None), self._h,
               "hiss_count")
        return out

    def join(self, eps, batch_bytes=0, mode=HISS_OUT_CSR, copy_to_host=False, on_batch=None):
        """Run the join; on_batch(hiss_batch) is called once per batch (raw
        struct, pointers valid during the call).  Returns the stats dict."""
        err = []

        def cb(user, bptr):
            try:
                on_batch(bptr.contents)
                return 0
            except BaseException as e:  # surfaced after the join returns
                err.append(e)
                return 1

        out = hiss_out(mode, 1 if copy_to_host else 0,
                       HISS_BATCH_FN(cb) if on_batch is not None else HISS_BATCH_FN(), None)
        rc = hiss_join(self._h, float(eps), int(batch_bytes), ctypes.byref(out))
        if err:
            raise err[0]
        _check(rc, self._h, "hiss_join")
        return self.stats()

    def _run(self, call, on_batch):
        err = []

        def cb(user, bptr):
            try:
                on_batch(bptr.contents)
                return 0
            except BaseException as e:  # surfaced after the call returns
                err.append(e)
                return 1

        fn = HISS_BATCH_FN(cb) if on_batch is not None else HISS_BATCH_FN()
        rc = call(fn)
        if err:
            raise err[0]
        return rc

    def join_shard(self, eps, rank, nranks, batch_bytes=0, mode=HISS_OUT_CSR, copy_to_host=False, on_batch=None):
        """Shard rank of nranks of the self-join (hiss_join_shard); on_batch as
        in ``join``.  Returns the stats dict."""
        def call(fn):
            out = hiss_out(mode, 1 if copy_to_host else 0, fn, None)
            return hiss_join_shard(self._h, float(eps), int(batch_bytes), ctypes.byref(out), int(rank), int(nranks))

        _check(self._run(call, on_batch), self._h, "hiss_join_shard")
        return self.stats()

    def join_shard_sets(self, eps, rank, nranks, batch_bytes=0):
        """Rows of one shard as {query id: numpy array of neighbour ids}."""
        res = {}

        def take(b):
            q = _host_array(b.query_ids, b.nq, np.int64)
            rp = _host_array(b.row_ptr, b.nq + 1, np.int64)
            cols = _host_array(b.cols, b.nnz, np.int32)
            for i in range(b.nq):
                res[int(q[i])] = cols[rp[i]:rp[i + 1]]

        self.join_shard(eps, rank, nranks, batch_bytes, HISS_OUT_CSR, True, take)
        return res

    def join_queries(self, queries, eps, batch_bytes=0, mode=HISS_OUT_CSR, copy_to_host=False, on_batch=None):
        """Semi-join of the query points (torch CUDA float32 (nq, d)) against
        the built dataset; on_batch as in ``join``.  Returns the stats dict."""
        q = queries.contiguous()
        assert q.is_cuda and q.dim() == 2 and q.shape[1] == self.d

        def call(fn):
            out = hiss_out(mode, 1 if copy_to_host else 0, fn, None)
            return hiss_join_queries(self._h, q.data_ptr() if q.numel() else None, q.shape[0], float(eps),
                                     int(batch_bytes), ctypes.byref(out))

        _check(self._run(call, on_batch), self._h, "hiss_join_queries")
        return self.stats()

    def join_queries_sets(self, queries, eps, batch_bytes=0):
        """Semi-join result as {query row: numpy array of data ids}."""
        res = {}

        def take(b):
            q = _host_array(b.query_ids, b.nq, np.int64)
            rp = _host_array(b.row_ptr, b.nq + 1, np.int64)
            cols = _host_array(b.cols, b.nnz, np.int32)
            for i in range(b.nq):
                res[int(q[i])] = cols[rp[i]:rp[i + 1]]

        self.join_queries(queries, eps, batch_bytes, HISS_OUT_CSR, True, take)
        return res

    def count_queries(self, queries, eps):
        import torch
        q = queries.contiguous()
        out = torch.empty(q.shape[0], dtype=torch.int64, device="cuda")
        _check(hiss_count_queries(self._h, q.data_ptr() if q.numel() else None, q.shape[0], float(eps),
                                  out.data_ptr() if q.numel() else None), self._h, "hiss_count_queries")
        return out

    def join_sets(self, eps, batch_bytes=0):
        """Full result as {query id: numpy array of neighbour ids}, through
        host delivery (copy_to_host = 1)."""
        res = {}

        def take(b):
            q = _host_array(b.query_ids, b.nq, np.int64)
            rp = _host_array(b.row_ptr, b.nq + 1, np.int64)
            cols = _host_array(b.cols, b.nnz, np.int32)
            for i in range(b.nq):
                res[int(q[i])] = cols[rp[i]:rp[i + 1]]

        self.join(eps, batch_bytes, HISS_OUT_CSR, True, take)
        return res

    def join_csr(self, eps, batch_bytes=0):
        """Full result as (row_ptr int64[n+1], cols int32[nnz]) in original
        query order, neighbours of each row sorted ascending (host arrays)."""
        rows = self.join_sets(eps, batch_bytes)
        n = self.n
        cnt = np.zeros(n + 1, dtype=np.int64)
        for q, c in rows.items():
            cnt[q + 1] = c.size
        row_ptr = np.cumsum(cnt)
        cols = np.empty(int(row_ptr[-1]), dtype=np.int32)
        for q, c in rows.items():
            cols[row_ptr[q]:row_ptr[q + 1]] = np.sort(c)
        return row_ptr, cols

    def index(self):
        v = hiss_index_view()
        _check(hiss_index(self._h, ctypes.byref(v)), self._h, "hiss_index")
        n, C = v.n, v.cells
        return {"n": n, "cells": C,
                "ids": _device_tensor(v.ids, n, "<i4"),
                "cell_start": _device_tensor(v.cell_start, C + 1, "<i4"),
                "cell_of_row": _device_tensor(v.cell_of_row, n, "<i4"),
                "nbr": _device_tensor(v.nbr, C * 27, "<i4"),
                "nbr_count": _device_tensor(v.nbr_count, C, "<i4"),
                "cell_bound": _device_tensor(v.cell_bound, C, "<i8"),
                "cell_key": _device_tensor(v.cell_key, C, "<i8"),
                "perm": list(v.perm), "sub_bits": v.sub_bits, "cell_width": v.cell_width,
                "origin": list(v.origin)}

    def stats(self):
        s = hiss_stats()
        _check(hiss_last_stats(self._h, ctypes.byref(s)), self._h, "hiss_last_stats")
        return {k: getattr(s, k) for k, _ in hiss_stats._fields_}

    def work_profile(self, eps):
        """(sum of per-pair early-exit dimensions, dimensions the join's
        refinement evaluates) over all candidate pairs for eps."""
        out = (_i64 * 2)()
        _check(hiss_work_profile(self._h, float(eps), out), self._h, "hiss_work_profile")
        return int(out[0]), int(out[1])

    def launches(self):
        return int(hiss_launch_count(self._h))

    def set_alloc_limit(self, nbytes):
        _check(hiss_set_option(self._h, HISS_OPT_ALLOC_LIMIT, int(nbytes)), self._h, "hiss_set_option")

    def knn(self, k, eps0=0.0):
        """Exact k nearest neighbours of every point (hiss_knn): (ids int64
        (n, k), squared distances float32 (n, k)) as torch CUDA tensors."""
        import torch
        ids = torch.empty((self.n, k), dtype=torch.int64, device="cuda")
        d2 = torch.empty((self.n, k), dtype=torch.float32, device="cuda")
        _check(hiss_knn(self._h, int(k), float(eps0), ids.data_ptr(), d2.data_ptr()), self._h, "hiss_knn")
        return ids, d2

    def set_refine(self, tensor_cores):
        """Select the refinement: CUDA cores (default) or the tensor-core
        prefilter with exact recheck (HISS_OPT_REFINE)."""
        mode = HISS_REFINE_TENSOR_CORES if tensor_cores else HISS_REFINE_CUDA_CORES
        _check(hiss_set_option(self._h, HISS_OPT_REFINE, mode), self._h, "hiss_set_option")
        return self

    # building blocks
    def sort_pairs(self, keys, vals, key_bits):
        _check(hiss_sort_pairs(self._h, keys.data_ptr(), vals.data_ptr(), keys.numel(), key_bits), self._h,
               "hiss_sort_pairs")

    def exclusive_scan(self, x, out):
        _check(hiss_exclusive_scan(self._h, x.data_ptr(), out.data_ptr(), x.numel()), self._h,
               "hiss_exclusive_scan")

    def mask_positions(self, words, nbits, pos):
        cnt = _i64()
        _check(hiss_mask_positions(self._h, words.data_ptr(), int(nbits), pos.data_ptr(), ctypes.byref(cnt)),
               self._h, "hiss_mask_positions")
        return int(cnt.value)
