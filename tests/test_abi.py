"""The C-ABI library builds for sm_103a, loads, and exports every entry point include/vc.h declares.
No compute calls: these run without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import LIB_PATH
    return ctypes.CDLL(LIB_PATH)


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(vc_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_round_calls():
    names = declared_symbols()
    for n in ["vc_compress_kv", "vc_draft_attn", "vc_verify_attn", "vc_accept", "vc_stage_full_kv",
              "vc_workspace_size", "vc_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.vc_status_string.restype = ctypes.c_char_p
    assert lib.vc_status_string(0) == b"ok"
    assert b"page-locked" in lib.vc_status_string(4)
    assert lib.vc_version() >= 100


def test_binding_names_match_header():
    import lossless_compressed_kv_vc_gb300 as vc
    for n in declared_symbols():
        assert hasattr(vc, n), n


def test_validation_rejects_without_launching(lib):
    """Host-side validation runs before any CUDA call, so it is testable without a GPU."""
    import lossless_compressed_kv_vc_gb300 as vc
    bad = vc.vc_shape(0, 8, 2, 64)
    assert vc.vc_draft_attn(bad, None, stream=0, raise_on_error=False) == vc.VC_ERR_INVALID
    shp = vc.vc_shape(1, 8, 2, 96)
    assert vc.vc_verify_attn(shp, None, stream=0, raise_on_error=False) in (vc.VC_ERR_INVALID, vc.VC_ERR_UNSUPPORTED)
    assert vc.vc_accept(0, 4, 10, 16, 16, 16, 16, 16, stream=0, raise_on_error=False) == vc.VC_ERR_INVALID
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, bad) == 0
    ok = vc.vc_shape(8, 32, 8, 128)
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, ok) > 0
