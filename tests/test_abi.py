"""The C-ABI library loads and exports every symbol include/sgemv.h
declares, and rejects bad arguments on the host before touching a GPU.
Runs without a GPU (no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_weight_only_gb300 as swo
from sparse_weight_only_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgemv.h")


@pytest.fixture(scope="module")
def lib():
    swo.build()
    return swo.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgemv_\w+)\s*\(", text)))


def test_header_declares_the_binding(lib):
    assert declared_functions() == sorted(_native.SIGNATURES)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", swo.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (sgemv_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def _create(lib, *args):
    h = ctypes.c_void_p()
    rc = lib.sgemv_create(ctypes.byref(h), *args)
    return rc, h


@pytest.mark.parametrize("args,needle", [
    ((64, 128, 3, 64, 1, 0), "n_keep"),
    ((64, 128, 0, 64, 1, 0), "n_keep"),
    ((64, 128, 2, 32, 1, 0), "group"),
    ((64, 192, 2, 128, 1, 0), "multiple"),
    ((64, 128, 2, 64, 0, 0), "max_m"),
    ((64, 128, 2, 64, 65, 0), "max_m"),
    ((-1, 128, 2, 64, 1, 0), "rows"),
    ((64, -64, 2, 64, 1, 0), "cols"),
    ((1 << 25, 128, 2, 64, 1, 0), "rows"),
    ((64, 1 << 21, 2, 64, 1, 0), "cols"),
])
def test_create_rejects_bad_arguments(lib, args, needle):
    rc, h = _create(lib, *args)
    assert rc == swo.SGEMV_ERR_ARG
    assert not h.value
    assert needle in lib.sgemv_last_error().decode()


def test_null_handle_calls(lib):
    assert lib.sgemv_destroy(None) == swo.SGEMV_OK
    assert lib.sgemv_packed_bytes(None) == 0
    for name, nargs in (("sgemv_pack", 1), ("sgemv_status", 0)):
        rc = getattr(lib, name)(None, *([None] * nargs))
        assert rc == swo.SGEMV_ERR_ARG
    assert lib.sgemv_run(None, None, None, 1, None) == swo.SGEMV_ERR_ARG
    assert lib.sgemv_run_host(None, None, None, 1, None) == swo.SGEMV_ERR_ARG
    # grouped runs: a negative count, NULL arrays, a NULL handle in the list
    for name in ("sgemv_run_group", "sgemv_run_group_host"):
        fn = getattr(lib, name)
        assert fn(None, -1, None, None, 1, None) == swo.SGEMV_ERR_ARG
        assert fn(None, 0, None, None, 1, None) == swo.SGEMV_OK       # count 0: no-op
        assert fn(None, 2, None, None, 1, None) == swo.SGEMV_ERR_ARG
        hs = (ctypes.c_void_p * 1)(None)
        ys = (ctypes.c_void_p * 1)(None)
        assert fn(hs, 1, None, ys, 1, None) == swo.SGEMV_ERR_ARG
    assert lib.sgemv_export(None, None, None, None, None) == swo.SGEMV_ERR_ARG
    assert lib.sgemv_import(None, None, None, None, None) == swo.SGEMV_ERR_ARG
    assert lib.sgemv_create(None, 1, 64, 2, 64, 1, 0) == swo.SGEMV_ERR_ARG
    assert "NULL" in lib.sgemv_last_error().decode()


def test_binding_refuses_missing_library(tmp_path):
    saved = _native._lib
    _native._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            _native.load(str(tmp_path / "libsgemv.so"))
    finally:
        _native._lib = saved
