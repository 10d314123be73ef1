"""The C ABI library loads, exports every entry point include/ar.h declares,
and rejects bad host-side arguments before making any CUDA call (so these
run without a GPU)."""
import ctypes
import os
import re

import pytest

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ar_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return ar.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ar_create", "ar_allreduce", "ar_ll_pack", "ar_ll_unpack", "ar_status",
                 "ar_destroy", "ar_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in ar.SIGNATURES, "binding lacks " + name


def test_binding_names_match_header():
    assert set(ar.SIGNATURES) == set(declared_functions())


def test_create_rejects_bad_arguments(lib):
    h = ctypes.c_void_p()
    for R, N, dt in [(0, 10, 0), (33, 10, 0), (-1, 10, 0), (4, 0, 0), (4, 10, 3), (4, 10, -1)]:
        assert lib.ar_create(R, N, dt, ctypes.byref(h)) == ar.AR_ERR_INVALID
    assert lib.ar_create(4, 10, 0, None) == ar.AR_ERR_INVALID


def test_null_handle_paths(lib):
    arr = (ctypes.c_void_p * 1)(0)
    assert lib.ar_allreduce(None, arr, arr, 0, 1, None) == ar.AR_ERR_INVALID
    assert lib.ar_reduce_scatter(None, arr, arr, None) == ar.AR_ERR_INVALID
    assert lib.ar_all_gather(None, arr, None) == ar.AR_ERR_INVALID
    assert lib.ar_ll_pack(None, None, None, 1, 1, None) == ar.AR_ERR_INVALID
    assert lib.ar_ll_unpack(None, None, None, 1, 1, None) == ar.AR_ERR_INVALID
    assert lib.ar_status(None, None) == ar.AR_ERR_INVALID
    assert lib.ar_set_timeout(None, 5) == ar.AR_ERR_INVALID
    assert lib.ar_debug_drop_rank(None, 0) == ar.AR_ERR_INVALID
    assert lib.ar_set_grid_divisor(None, 1) == ar.AR_ERR_INVALID
    out = ctypes.c_int(0)
    assert lib.ar_get_grid_divisor(None, 16, 0, 1, ctypes.byref(out)) == ar.AR_ERR_INVALID
    assert lib.ar_get_info(None, None) == ar.AR_ERR_INVALID
    assert lib.ar_destroy(None) == ar.AR_OK


def test_round_rejects_bad_arguments(lib):
    assert lib.ar_round(7, 16, 16, 1, None) == ar.AR_ERR_INVALID
    assert lib.ar_round(0, None, 16, 1, None) == ar.AR_ERR_INVALID
    assert lib.ar_round(0, 18, 16, 1, None) == ar.AR_ERR_INVALID     # src not 4-byte aligned
    assert lib.ar_round(2, 16, 18, 1, None) == ar.AR_ERR_INVALID     # fp32 dst misaligned


def test_strerror_names_every_code(lib):
    for code in range(0, 7):
        s = ar.ar_strerror(code)
        assert s.startswith("AR_")
    assert "unknown" in ar.ar_strerror(99)


def test_library_is_sm103a_only():
    assert cuda_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        ar.load_library(str(tmp_path / "absent.so"))
