"""The C-ABI library loads and exports every function include/bi.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(bi_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from invariant_fixed_order_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("bi_rmsnorm", "bi_gemm", "bi_decode_attention", "bi_prefill_attention", "bi_argmax",
              "bi_forward_step", "bi_model_create", "bi_model_destroy", "bi_forward_workspace_size",
              "bi_last_error", "bi_check_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls(lib):
    lib.bi_version.restype = ctypes.c_int32
    assert lib.bi_version() >= 1
    lib.bi_last_error.restype = ctypes.c_char_p
    lib.bi_rope_table.restype = ctypes.c_int32
    lib.bi_rope_table.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double]
    # validation happens before anything touches the device
    assert lib.bi_rope_table(None, None, 4, 64, 500000.0) == 1  # BI_ERR_INVALID
    assert b"null" in lib.bi_last_error()
    lib.bi_gemm_workspace_size.restype = ctypes.c_size_t
    lib.bi_gemm_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    assert lib.bi_gemm_workspace_size(64, 4096, 4096, 0) == 0  # invariant mode needs no workspace
