"""The C-ABI library on the host (no GPU): it loads, exports every entry
point include/hc_read.h and include/hc_q2.h declare, and rejects bad arguments before touching
the device."""

import ctypes
import os
import re

import pytest

import hyper_connection_residual_gb300 as hc
from hyper_connection_residual_gb300 import build as hcbuild

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, name) for name in ("hc_read.h", "hc_q2.h")]


@pytest.fixture(scope="module")
def lib():
    hcbuild.build()
    return hc.load()


def declared_functions():
    src = ""
    for path in HEADERS:
        with open(path) as f:
            src += f.read()
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
    assert lib.hc_read_set_wait_limit(None, 5) == hc.HC_ERR_ARG
    assert lib.hc_read_set_overlap(None, 1) == hc.HC_ERR_ARG
    assert lib.hc_read_down_tiles_bytes(None) == -1
    assert lib.hc_read_register_down_tiles(None, None, None, None) == hc.HC_ERR_ARG
    assert lib.hc_read_forget_down_tiles(None, None) == hc.HC_ERR_ARG
    assert lib.hc_read_up_tiles_bytes(None) == -1
    assert lib.hc_read_register_up_tiles(None, None, None, None) == hc.HC_ERR_ARG
    assert lib.hc_read_forget_up_tiles(None, None) == hc.HC_ERR_ARG


def test_q2_matvec_rejects_bad_arguments(lib):
    """hc_q2_0_matvec validates on the host before any CUDA call: the pointers
    below are never dereferenced (distinct 16-byte-aligned fake addresses,
    ranges far apart)."""
    rows, cols, ncols = 12288, 2560, 2
    Wq, Ws, x, y = 1 << 40, 2 << 40, 3 << 40, 4 << 40
    f = lib.hc_q2_0_matvec
    assert f(None, Ws, rows, cols, x, ncols, y, None) == hc.HC_ERR_ARG
    assert f(Wq, None, rows, cols, x, ncols, y, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, rows, cols, None, ncols, y, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, rows, cols, x, ncols, None, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, 0, cols, x, ncols, y, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, (1 << 24) + 1, cols, x, ncols, y, None) == hc.HC_ERR_ARG
    for bad in (0, 5, -1):
        assert f(Wq, Ws, rows, cols, x, bad, y, None) == hc.HC_ERR_ARG
    for bad in (256, 2560 + 64, 2560 + 256, 4096 + 512, 16384, 0, -512):
        assert f(Wq, Ws, rows, bad, x, ncols, y, None) == hc.HC_ERR_SHAPE
    for i in range(4):
        ptrs = [Wq, Ws, x, y]
        ptrs[i] += 8
        assert f(ptrs[0], ptrs[1], rows, cols, ptrs[2], ncols, ptrs[3], None) == hc.HC_ERR_ALIGN
    # y overlapping an input
    assert f(Wq, Ws, rows, cols, x, ncols, Wq + 16, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, rows, cols, x, ncols, Ws + 64 * 12288 - 16, None) == hc.HC_ERR_ARG
    assert f(Wq, Ws, rows, cols, x, ncols, x - 16, None) == hc.HC_ERR_ARG


def test_q2_batch_rejects_bad_arguments(lib):
    """hc_q2_0_matvec_batch checks every product before enqueuing anything."""
    rows, cols, ncols = 12288, 2560, 2
    D = hc.hc_q2_0_desc
    good = [D(1 << 40, 2 << 40, 3 << 40, 4 << 40), D(5 << 40, 6 << 40, 3 << 40, 7 << 40)]
    f = lib.hc_q2_0_matvec_batch

    def arr(items):
        a = (D * len(items))()
        for j, d in enumerate(items):
            a[j] = d
        return a

    assert f(None, 1, rows, cols, ncols, None) == hc.HC_ERR_ARG
    assert f(arr(good), 0, rows, cols, ncols, None) == hc.HC_ERR_ARG
    assert f(arr(good), 2, rows, 2560 + 64, ncols, None) == hc.HC_ERR_SHAPE
    assert f(arr(good), 2, rows, cols, 5, None) == hc.HC_ERR_ARG
    bad = [good[0], D(5 << 40, 6 << 40, None, 7 << 40)]
    assert f(arr(bad), 2, rows, cols, ncols, None) == hc.HC_ERR_ARG
    bad = [good[0], D(5 << 40, (6 << 40) + 4, 3 << 40, 7 << 40)]
    assert f(arr(bad), 2, rows, cols, ncols, None) == hc.HC_ERR_ALIGN
    bad = [good[0], D(5 << 40, 6 << 40, 3 << 40, 5 << 40)]     # y over its own codes
    assert f(arr(bad), 2, rows, cols, ncols, None) == hc.HC_ERR_ARG
