"""The C-ABI library builds for sm_103a, loads, and exports every entry
point include/hiss.h declares (no compute call: runs without a GPU)."""
import ctypes
import importlib.util
import os
import re

from conftest import ROOT


def _builder():
    path = os.path.join(ROOT, "exact_dimensional_distance_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_hiss_build_t", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "hiss.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(hiss_\w+)\s*\(", src, flags=re.M))


def test_library_exports_every_declared_symbol():
    lib_path = _builder().build()
    lib = ctypes.CDLL(lib_path)
    names = _declared()
    assert {"hiss_create", "hiss_build", "hiss_count", "hiss_join", "hiss_destroy"} <= names
    for name in sorted(names):
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    _builder().build()
    import exact_dimensional_distance_gb300 as edd
    assert set(edd.EXPORTED) == _declared()
    for name in edd.EXPORTED:
        assert callable(getattr(edd, name))


def test_struct_sizes_match_header_layout():
    import exact_dimensional_distance_gb300 as edd
    # int64 x10, int32 x4, float, double x8 (with one 4-byte pad before the first double)
    assert ctypes.sizeof(edd.hiss_stats) == 10 * 8 + 4 * 4 + 4 + 4 + 8 * 8
    assert ctypes.sizeof(edd.hiss_batch) == 10 * 8 + 2 * 4
