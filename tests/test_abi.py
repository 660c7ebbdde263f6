"""The C ABI library builds, loads and exports what include/specverify.h declares.

No compute calls here: on a host without a GPU only argument checking and the
"no device" error path are exercised.
"""
import ctypes

import pytest

from speculative_decoding_verification_10_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_every_declared_function_is_exported(lib):
    names = _lib.header_functions()
    assert {"specverify_create", "specverify_run", "specverify_destroy",
            "specverify_status", "specverify_error_string"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, 17):
        assert isinstance(_lib.error_string(code), str)
    assert _lib.error_string(-4) == "handle already destroyed"


def test_create_rejects_bad_arguments_before_touching_cuda(lib):
    h = ctypes.c_void_p()
    assert lib.specverify_create(None, 0, 8, 3, 1024, 1) == _lib.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 8, 3, 1024, 7) == _lib.ERR_DTYPE
    assert lib.specverify_create(ctypes.byref(h), 0, 0, 3, 1024, 1) == _lib.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 4097, 3, 1024, 1) == _lib.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 8, 32, 1024, 1) == _lib.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 8, 3, 0, 1) == _lib.ERR_INVALID_ARG
    assert lib.specverify_create_ex(ctypes.byref(h), 0, 8, 3, 1024, 1, 8) == _lib.ERR_INVALID_ARG
    assert h.value is None


def test_calls_on_a_null_handle(lib):
    st = ctypes.c_int32()
    assert lib.specverify_status(None, ctypes.byref(st)) == _lib.ERR_INVALID_ARG
    assert lib.specverify_destroy(None) == _lib.ERR_INVALID_ARG
    assert lib.specverify_run(None, None, None, None, None, None, 0, 1, 0,
                              None, None, None, None) == _lib.ERR_INVALID_ARG
    n = ctypes.c_int(-7)
    assert lib.specverify_launches_per_run(None, 4, ctypes.byref(n)) == _lib.ERR_INVALID_ARG
    assert lib.specverify_set_depth(None, 1) == _lib.ERR_INVALID_ARG
    assert n.value == -7


def test_no_device_reports_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.specverify_create(ctypes.byref(h), 0, 8, 3, 1024, 1) == _lib.ERR_CUDA


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        _lib.load(str(tmp_path / "missing.so"))


def test_static_entry_rejects_inputs_above_its_limits(lib):
    # checked before any device call: nothing is launched, nothing allocated
    args = [None] * 5
    big = lib.specverify_run_static(0, 3, 1024, 1, *args, 1, _lib.STATIC_MAX_BATCH + 1, 0,
                                    None, None, None, None)
    assert big == _lib.ERR_TOO_LARGE
    deep = lib.specverify_run_static(0, _lib.STATIC_MAX_K + 1, 1024, 1, *args, 1, 4, 0,
                                     None, None, None, None)
    assert deep == _lib.ERR_TOO_LARGE
    assert lib.specverify_run_static(0, 3, 1024, 9, *args, 1, 4, 0,
                                     None, None, None, None) == _lib.ERR_DTYPE
    assert b"static scratch limits" in lib.specverify_error_string(_lib.ERR_TOO_LARGE)
