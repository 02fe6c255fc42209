"""The C ABI library loads without a GPU and exports every declared entry point.

No compute call is made here: only calls that return before touching CUDA
(version, status text, argument validation).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ts_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from token_level_sparse_gb300 import build
    build.build()
    import token_level_sparse_gb300 as T
    return T.library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["ts_create", "ts_destroy", "ts_cache_create", "ts_cache_destroy", "ts_cache_reset",
                 "ts_cache_check", "ts_score", "ts_select", "ts_sparse_attend", "ts_decode_step",
                 "ts_get_status", "ts_status_str", "ts_version"]:
        assert want in names, want


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings_and_version(lib):
    import token_level_sparse_gb300 as T
    assert T.ts_version() == 100
    for code in T.STATUS:
        assert T.ts_status_str(code) and T.ts_status_str(code) != "unknown status"
    assert T.ts_status_str(999) == "unknown status"


def test_validation_before_cuda(lib):
    import token_level_sparse_gb300 as T
    INVALID = T.STATUS_CODE["TS_ERR_INVALID_ARG"]
    assert lib.ts_create(None, None) == INVALID
    h = ctypes.c_void_p()
    assert lib.ts_create(ctypes.byref(h), None) == INVALID
    bad = T.Config(32, 5, 128, 16, T.TS_KV_BF16, 1, 10, 10)       # H not a multiple of H_kv
    assert lib.ts_create(ctypes.byref(h), ctypes.byref(bad)) == INVALID
    odd_page = T.Config(32, 8, 128, 8, T.TS_KV_BF16, 1, 10, 10)
    assert lib.ts_create(ctypes.byref(h), ctypes.byref(odd_page)) == T.STATUS_CODE["TS_ERR_UNSUPPORTED"]
    # one token per page passes validation (here, without a GPU, creation then stops at CUDA), and
    # its token count is bounded like 16-token pages'
    token_pages = T.Config(32, 8, 128, 1, T.TS_KV_BF16, 1, 10, 10)
    rc = lib.ts_create(ctypes.byref(h), ctypes.byref(token_pages))
    assert rc not in (T.STATUS_CODE["TS_ERR_UNSUPPORTED"], INVALID, T.STATUS_CODE["TS_ERR_SHAPE"])
    if rc == 0:                                     # (with a GPU the context exists)
        lib.ts_destroy(h)
    too_many = T.Config(32, 8, 128, 1, T.TS_KV_BF16, 1, (1 << 30) + 1, 10)
    assert lib.ts_create(ctypes.byref(h), ctypes.byref(too_many)) == T.STATUS_CODE["TS_ERR_SHAPE"]
    no_kernel = T.Config(24, 8, 96, 16, T.TS_KV_BF16, 1, 10, 10)
    assert lib.ts_create(ctypes.byref(h), ctypes.byref(no_kernel)) == T.STATUS_CODE["TS_ERR_UNSUPPORTED"]
    p = T.params()
    assert lib.ts_score(None, None, None, None, None, 1, None, 0.0, None, 0, None) == INVALID
    assert lib.ts_select(None, None, 0, None, None, 0, None, 1, None, ctypes.byref(p), None, 0, None,
                         None) == INVALID
    assert lib.ts_sparse_attend(None, None, None, None, None, None, 0, None, 1, 0.0, None, None,
                                None) == INVALID
    assert lib.ts_decode_step(None, None, 0, None, None, None, None, None, 1, ctypes.byref(p), None, 0,
                              None, 0, None, None, None, None, None) == INVALID
    v = ctypes.c_int()
    assert lib.ts_get_status(None, ctypes.byref(v), None) == INVALID
    assert lib.ts_cache_create(None, ctypes.byref(h), 1, 1) == INVALID


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import token_level_sparse_gb300 as T
    monkeypatch.setattr(T, "_lib", None)
    monkeypatch.setattr(T, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        T.library()
