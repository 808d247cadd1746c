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


def test_struct_layouts_match_header(tmp_path):
    # the binding's ctypes structures against the C compiler's layout of hiss.h
    import shutil
    import subprocess
    import pytest
    import exact_dimensional_distance_gb300 as edd
    if shutil.which("gcc") is None:
        pytest.skip("needs gcc")
    structs = {"hiss_stats": edd.hiss_stats, "hiss_batch": edd.hiss_batch, "hiss_out": edd.hiss_out,
               "hiss_index_view": edd.hiss_index_view}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "hiss.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (name, name))
        for field, _ in cls._fields_:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (name, field, name, field))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I" + os.path.join(ROOT, "include"), "-o", str(exe), str(src)])
    got = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        a, b, v = line.split()
        got[(a, b)] = int(v)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)
