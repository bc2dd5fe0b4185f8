"""The C-ABI library on the host (no GPU): it loads, exports every entry
point include/hc_read.h declares, and rejects bad arguments before touching
the device."""

import ctypes
import os
import re

import pytest

import hyper_connection_residual_gb300 as hc
from hyper_connection_residual_gb300 import build as hcbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "hc_read.h")


@pytest.fixture(scope="module")
def lib():
    hcbuild.build()
    return hc.load()


def declared_functions():
    with open(HEADER) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|void|int64_t|const char\*)\s+(hc_\w+)\s*\(", src, re.M)))


def test_header_matches_binding_exports():
    assert declared_functions() == sorted(hc.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.hc_status_str(code)
    assert hc.status_str(-3) == "geometry not supported"


def test_create_rejects_unsupported_geometry(lib):
    h = ctypes.c_void_p()
    assert lib.hc_read_create(ctypes.byref(h), 4, 2048, 320, 8, 1e-6, 0) == hc.HC_ERR_SHAPE
    assert lib.hc_read_create(ctypes.byref(h), 2, 2560, 320, 8, 1e-6, 0) == hc.HC_ERR_SHAPE
    assert lib.hc_read_create(ctypes.byref(h), 4, 2560, 320, 0, 1e-6, 0) == hc.HC_ERR_ARG
    assert lib.hc_read_create(ctypes.byref(h), 4, 2560, 320, 65, 1e-6, 0) == hc.HC_ERR_ARG
    assert lib.hc_read_create(ctypes.byref(h), 4, 2560, 320, 8, -1.0, 0) == hc.HC_ERR_ARG
    assert lib.hc_read_create(None, 4, 2560, 320, 8, 1e-6, 0) == hc.HC_ERR_ARG
    assert h.value is None


def test_null_handle_rejected(lib):
    assert lib.hc_read(None, *([None] * 6), 1, *([None] * 3), None) == hc.HC_ERR_ARG
    assert lib.hc_read_check(None) == hc.HC_ERR_ARG
    assert lib.hc_read_reset(None, None) == hc.HC_ERR_ARG
    assert lib.hc_read_scratch_bytes(None) == -1
    lib.hc_read_destroy(None)
    assert lib.hc_graph_launch(None, None) == hc.HC_ERR_ARG
    assert lib.hc_graph_end(None, None) == hc.HC_ERR_ARG
    assert lib.hc_read_q8(None, *([None] * 8), 1, *([None] * 6)) == hc.HC_ERR_ARG
