"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/tovl.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re
import subprocess

import pytest

from consumer_movement_gemm_gb300 import build as tovl_build
from consumer_movement_gemm_gb300 import tovl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tovl.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tovl_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    tovl_build.build()
    return tovl.load()


def test_header_declares_the_four_entry_points():
    names = _declared_functions()
    for n in ["tovl_create", "tovl_gather_gemm", "tovl_dispatch_grouped_gemm", "tovl_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", tovl.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    # the binding describes every declared function, with no extras
    assert sorted(tovl.SIGNATURES) == _declared_functions()
    # internal launchers stay hidden
    assert not [n for n in exported if "launch" in n]


def test_error_strings(lib):
    assert tovl.error_string(0) == "ok"
    assert "timed out" in tovl.error_string(4)


def test_dispatch_rows_closed_form(lib):
    for T, k, E in [(4096, 2, 8), (8192, 4, 32), (1, 1, 1), (0, 2, 3)]:
        want = -(-(T * k + E * 127) // 128) * 128
        assert tovl.dispatch_rows(T, k, E) == want


def test_dispatch_rows_aligned_closed_form(lib):
    for T, k, E in [(4096, 2, 8), (8192, 4, 32), (1, 1, 1), (0, 2, 3)]:
        assert tovl.dispatch_rows_aligned(T, k, E, 128) == tovl.dispatch_rows(T, k, E)
        want = -(-(T * k + E * 255) // 256) * 256
        assert tovl.dispatch_rows_aligned(T, k, E, 256) == want
    assert tovl.dispatch_rows_aligned(10, 2, 3, 192) == 0       # only 128 and 256
    assert tovl.dispatch_rows_aligned(-1, 2, 3, 128) == 0


def test_new_entry_points_reject_null_handles(lib):
    L = tovl.load()
    assert L.tovl_combine(None, None, 0, None, None, None, None) == tovl.TOVL_ERR_INVALID
    assert L.tovl_gemm_reduce_scatter(None, None, 0, 0, 0, None, 0, None, None, None) == tovl.TOVL_ERR_INVALID
    v = ctypes.c_longlong()
    for opt in (14, 15, 16, 17, 18, 19, 20, 23):
        assert L.tovl_set_option(None, opt, 0) == tovl.TOVL_ERR_INVALID
        assert L.tovl_get_option(None, opt, ctypes.byref(v)) == tovl.TOVL_ERR_INVALID


def test_host_argument_errors(lib):
    L = tovl.load()
    assert L.tovl_create(None, None) == tovl.TOVL_ERR_INVALID
    h = ctypes.c_void_p()
    assert L.tovl_create(ctypes.byref(h), None) == tovl.TOVL_ERR_INVALID
    cfg = tovl.default_config(0)
    cfg.chunk_rows = 32
    assert L.tovl_create(ctypes.byref(h), ctypes.byref(cfg)) == tovl.TOVL_ERR_UNSUPPORTED
    assert L.tovl_destroy(None) == tovl.TOVL_OK
    assert L.tovl_sync_status(None) == tovl.TOVL_ERR_INVALID
    assert L.tovl_gather_gemm(None, None, 0, 0, 0, None, 0, None, None, None) == tovl.TOVL_ERR_INVALID


def test_create_without_gpu_is_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    cfg = tovl.default_config(0)
    assert tovl.load().tovl_create(ctypes.byref(h), ctypes.byref(cfg)) == tovl.TOVL_ERR_UNSUPPORTED
    assert not h.value


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(tovl.TovlError):
        # a fresh loader state pointed at a path with no library
        saved = tovl._lib
        tovl._lib = None
        try:
            tovl.load(str(tmp_path / "libtovl.so"))
        finally:
            tovl._lib = saved
