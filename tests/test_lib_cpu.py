"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a GPU,
exports every entry point include/gocr.h declares, and its host-side argument
checks reject bad calls before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from self_speculative_block_gb300 import build, gocr
    build.build()
    return gocr.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gocr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(gocr_[a-z_0-9]+)\s*\(", src))
    return sorted(n for n in names if not n.endswith("_fn"))


def test_header_declares_the_boundary_calls():
    names = declared_symbols()
    for n in ("gocr_create", "gocr_prefill", "gocr_decode", "gocr_free"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from self_speculative_block_gb300 import gocr
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(declared_symbols()) == set(gocr.EXPORTS)


def test_create_rejects_bad_shapes_on_the_host(lib):
    from self_speculative_block_gb300 import gocr
    c = gocr.Config(2, 100, 4, 2, 64, 704, 1024, 0, 1e-6, 1e4, 128, 8, 1, -1)  # hidden % 128 != 0
    w = gocr.Weights()
    h = ctypes.c_void_p()
    rc = lib.gocr_create(ctypes.byref(c), ctypes.byref(w), None, gocr.ALLOC_FN(), gocr.FREE_FN(), None,
                         ctypes.byref(h))
    assert rc == -1 and not h.value
    assert "shape" in gocr.last_error(None)


def test_null_handle_calls_fail_cleanly(lib):
    out = np.zeros(4, np.int32)
    assert lib.gocr_decode(None, 0, 0, 0, 4, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), None) == -1
    assert lib.gocr_prefill(None, 0, None, 4) == -1
    lib.gocr_free(None)


def test_op_entry_points_validate_arguments(lib):
    assert lib.gocr_op_linear_workspace(0, 128, 128) == 0
    assert lib.gocr_op_linear_workspace(33, 256, 1536) > 0
    assert lib.gocr_op_linear(0, None, None, None, 1, 1, 8, None, 0, None) == -1
    assert lib.gocr_op_linear_planes(None, None, None, None, 1, 1, 8, None, 0, 0, None) == -1
    one = ctypes.c_void_p(16)
    assert lib.gocr_op_linear_planes(one, ctypes.c_void_p(18), one, one, 1, 1, 8, one, 1 << 20, 0, None) == -1
    assert b"aligned" in lib.gocr_last_error(None)
    assert lib.gocr_op_linear_planes(one, one, one, one, 1, 1, 8, one, 1 << 20, 6, None) == -1
    assert b"flags" in lib.gocr_last_error(None)
    assert lib.gocr_op_attention(1, None, None, None, None, None, None, None, None, 1, 4, 2, 64, 16, None) == -1


def test_split_rule_depends_on_n_and_k_only(lib):
    # The workspace formula is linear in T for fixed (N, K): same split count for any T.
    a = lib.gocr_op_linear_workspace(1, 2560, 1536)
    b = lib.gocr_op_linear_workspace(65, 2560, 1536)
    c = lib.gocr_op_linear_workspace(129, 2560, 1536)
    # (b - a) and (c - b) are the partial-buffer growth of 64 rows, plus counter padding
    assert abs((c - b) - (b - a)) <= 512
