"""The C-ABI library builds, loads without a GPU and exports every symbol
include/zsolve.h declares.  Only host-side entry points are called."""
import ctypes
import re

import mixed_precision_refinement_gb300 as zs


def test_library_exports_every_declared_symbol():
    names = zs.declared_symbols()
    assert len(names) >= 17
    lib = ctypes.CDLL(zs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    for n in zs.declared_symbols():
        assert callable(getattr(zs, n)), n


def test_header_documents_status_codes():
    for code in range(0, -8, -1):
        s = zs.zsolve_strerror(code)
        assert s and s != "unknown status"
    assert zs.zsolve_strerror(-99) == "unknown status"


def test_default_opts():
    o = zs.zsolve_default_opts()
    assert o.tol == 1e-11 and o.max_iter == 10 and o.outer_block == 128 and o.batch == 0
    assert o.force_fallback == 0


def test_create_rejects_bad_arguments_without_touching_the_device():
    lib = zs.raw_lib()
    ctx = ctypes.c_void_p()
    assert lib.zsolve_create(ctypes.byref(ctx), 0, 1, None) == zs.ZSOLVE_EINVAL
    assert lib.zsolve_create(ctypes.byref(ctx), 10, 0, None) == zs.ZSOLVE_EINVAL
    bad = zs.zsolve_default_opts()
    bad.outer_block = 64
    assert lib.zsolve_create(ctypes.byref(ctx), 10, 1, ctypes.byref(bad)) == zs.ZSOLVE_EINVAL
    assert lib.zsolve_create(None, 10, 1, None) == zs.ZSOLVE_EINVAL


def test_header_entry_points_cite_or_explain():
    text = open(zs.HEADER).read()
    assert "Solving Dense Matrices Fast in the Browser" in text
    for name in zs.declared_symbols():
        assert re.search(r"\b" + name + r"\s*\(", text)
