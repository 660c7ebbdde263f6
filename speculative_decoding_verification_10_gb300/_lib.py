"""ctypes view of libspecverify.so (the C ABI of include/specverify.h).

The library is loaded from the package's in-tree _build directory.  There is
no fallback: if the shared library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

HEADER = os.path.join(_build.INCLUDE, "specverify.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_DTYPE = -2
ERR_CUDA = -3
ERR_DESTROYED = -4
ERR_NO_STAGING = -5
ERR_TOO_LARGE = -6

SCHEDULE_AUTO = 0
SCHEDULE_WAVES = 1

HOST_READS_AUTO = 0
HOST_READS_STAGE = 1

STATIC_MAX_BATCH = 256
STATIC_MAX_K = 7

STATUS_BAD_TOKEN = 1
STATUS_BAD_K = 2
STATUS_BAD_TEMP = 4
STATUS_NONFINITE = 8
STATUS_BAD_TOTAL = 16
STATUS_BAD_PARENT = 32
STATUS_NO_DRAFT = 64
STATUS_BAD_CONF = 512
STATUS_BAD_TRUNC = 1024

CREATE_HOST_STAGING = 1

DTYPE_F32 = 0
DTYPE_BF16 = 1

_lib = None


def header_functions():
    """Names of the functions include/specverify.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char \*)\s*(specverify_\w+)\s*\(",
                                 text, flags=re.M)))


def load(path: str | None = None):
    """Load (once) and return the CDLL with argument types set."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"libspecverify.so not found at {path}; build it with "
            "speculative_decoding_verification_10_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.specverify_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I]
    lib.specverify_create.restype = I
    lib.specverify_create_ex.argtypes = [ctypes.POINTER(P), I, I, I, I, I, ctypes.c_uint]
    lib.specverify_create_ex.restype = I
    lib.specverify_run.argtypes = [P, P, P, P, P, P, ctypes.c_uint64, I, I, P, P, P, P]
    lib.specverify_run.restype = I
    lib.specverify_run_ex.argtypes = [P, P, P, P, P, P, ctypes.c_uint64, I, I, P, P, P,
                                      P, P, P, P, P, P]
    lib.specverify_run_ex.restype = I
    lib.specverify_run_host.argtypes = [P, P, P, P, P, P, ctypes.c_uint64, I, I, P, P, P, P]
    lib.specverify_run_host.restype = I
    lib.specverify_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.specverify_status.restype = I
    lib.specverify_set_timing_events.argtypes = [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]
    lib.specverify_set_timing_events.restype = I
    lib.specverify_launches_per_run.argtypes = [P, I, ctypes.POINTER(ctypes.c_int)]
    lib.specverify_launches_per_run.restype = I
    lib.specverify_run_static.argtypes = [I, I, I, I, P, P, P, P, P, ctypes.c_uint64, I, I,
                                          P, P, P, P]
    lib.specverify_run_static.restype = I
    lib.specverify_debug_set_epoch.argtypes = [P, ctypes.c_uint32]
    lib.specverify_debug_set_epoch.restype = I
    lib.specverify_static_debug_set_epoch.argtypes = [I, ctypes.c_uint32]
    lib.specverify_static_debug_set_epoch.restype = I
    lib.specverify_set_schedule.argtypes = [P, I]
    lib.specverify_set_schedule.restype = I
    lib.specverify_set_depth.argtypes = [P, I]
    lib.specverify_set_depth.restype = I
    lib.specverify_set_host_reads.argtypes = [P, I]
    lib.specverify_set_host_reads.restype = I
    lib.specverify_wave_depth.argtypes = [P, I, ctypes.POINTER(I)]
    lib.specverify_wave_depth.restype = I
    lib.specverify_last_host_reads.argtypes = [P, ctypes.POINTER(I)]
    lib.specverify_last_host_reads.restype = I
    lib.specverify_metrics.argtypes = [P, P, I, I, P, P, P, P, P]
    lib.specverify_metrics.restype = I
    lib.specverify_run_truncated.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_uint64, I, I,
                                             P, P, P, P]
    lib.specverify_run_truncated.restype = I
    lib.specverify_run_trimmed.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_uint64, I, I,
                                           P, P, P, P, P, P, P, P, P]
    lib.specverify_run_trimmed.restype = I
    lib.specverify_truncate.argtypes = [I, I, P, P, P, P, P, P, I, I, P, P, P, P]
    lib.specverify_truncate.restype = I
    lib.specverify_tree_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I]
    lib.specverify_tree_create.restype = I
    lib.specverify_tree_run.argtypes = [P, P, P, P, P, I, I, P, P, P, P, P]
    lib.specverify_tree_run.restype = I
    lib.specverify_tree_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.specverify_tree_status.restype = I
    lib.specverify_tree_destroy.argtypes = [P]
    lib.specverify_tree_destroy.restype = I
    lib.specverify_destroy.argtypes = [P]
    lib.specverify_destroy.restype = I
    lib.specverify_error_string.argtypes = [I]
    lib.specverify_error_string.restype = ctypes.c_char_p
    if path == _build.LIB_PATH:
        _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().specverify_error_string(code).decode()
