"""ctypes binding of libsmla.so: argument marshalling only.

Loads the in-tree ``libsmla.so`` (built by ``sparse_mla_attention_gb300.build``)
and declares the signatures of every entry point of ``include/smla.h``.
There is no fallback: if the library is missing, loading raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB

# Status codes (include/smla.h, enum smla_status).
SMLA_OK = 0
SMLA_ERR_NULL = 1
SMLA_ERR_SHAPE = 2
SMLA_ERR_D512 = 3
SMLA_ERR_NUM_KV_LT_T = 4
SMLA_ERR_RCHUNK = 5
SMLA_ERR_ALIGN = 6
SMLA_ERR_OVERLAP = 7
SMLA_ERR_WORKSPACE = 8
SMLA_ERR_ARCH = 9
SMLA_ERR_CUDA = 10
SMLA_ERR_INDEX = 11
SMLA_ERR_TIMEOUT = 12
SMLA_ERR_SINK = 13
SMLA_ERR_ARG = 14
SMLA_ERR_DEVICE = 15

SMLA_OP_FWD, SMLA_OP_BWD, SMLA_OP_CSR, SMLA_OP_BWD_HOST = 0, 1, 2, 3

EXPORTED = ("smla_workspace_size", "smla_fwd", "smla_bwd", "smla_bwd_host", "smla_csr_build",
            "smla_get_device_status", "smla_status_string", "smla_version",
            "smla_profiling", "smla_profile_read", "smla_dsink_static",
            "smla_selftest_wait_timeout", "smla_bwd_partial", "smla_reduce_partials")


class SmlaDims(ctypes.Structure):
    """Mirror of ``smla_dims``."""

    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("num_kv", ctypes.c_int32),
                ("r_chunk", ctypes.c_int32), ("scale", ctypes.c_float)]


class SmlaPhaseStat(ctypes.Structure):
    """Mirror of ``smla_phase_stat``."""

    _fields_ = [("name", ctypes.c_char_p), ("total_ms", ctypes.c_double),
                ("calls", ctypes.c_longlong), ("launches", ctypes.c_longlong)]


class SmlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libsmla.so and declare its signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise OSError(f"{path} not found: build it with "
                          "`python -m sparse_mla_attention_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
        dims_p = ctypes.POINTER(SmlaDims)
        lib.smla_workspace_size.argtypes = [ctypes.c_int, dims_p, ctypes.POINTER(sz)]
        lib.smla_fwd.argtypes = [vp] * 6 + [dims_p, vp, sz, vp]
        lib.smla_bwd.argtypes = [vp] * 10 + [dims_p, vp, sz, vp]
        lib.smla_bwd_host.argtypes = [vp] * 10 + [dims_p, vp, sz, vp]
        lib.smla_bwd_partial.argtypes = [vp] * 10 + [dims_p, vp, sz, vp]
        lib.smla_reduce_partials.argtypes = [vp, i32, ctypes.c_int64, vp, vp, vp]
        lib.smla_csr_build.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
        lib.smla_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        lib.smla_dsink_static.argtypes = [vp] * 5 + [i32, i32, vp]
        lib.smla_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint32, vp]
        lib.smla_profiling.argtypes = [ctypes.c_int]
        lib.smla_profile_read.argtypes = [ctypes.POINTER(SmlaPhaseStat), ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int)]
        lib.smla_status_string.argtypes = [ctypes.c_int]
        lib.smla_status_string.restype = ctypes.c_char_p
        for name in ("smla_workspace_size", "smla_fwd", "smla_bwd", "smla_bwd_host", "smla_csr_build",
                     "smla_get_device_status", "smla_version", "smla_profiling",
                     "smla_profile_read", "smla_dsink_static", "smla_selftest_wait_timeout",
                     "smla_bwd_partial", "smla_reduce_partials"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    try:
        return load().smla_status_string(int(code)).decode()
    except OSError:
        return f"status {code}"


def check(code: int, where: str) -> None:
    if code != SMLA_OK:
        raise SmlaError(code, where)


def profiling(enable: bool) -> None:
    """Turn the library's phase profiler on (and reset it) or off."""
    check(load().smla_profiling(1 if enable else 0), "smla_profiling")


def profile_read() -> dict:
    """{phase: {"ms": total, "calls": n, "launches": kernels}} since the last reset."""
    lib = load()
    arr = (SmlaPhaseStat * 16)()
    n = ctypes.c_int(0)
    check(lib.smla_profile_read(arr, 16, ctypes.byref(n)), "smla_profile_read")
    return {arr[i].name.decode(): {"ms": arr[i].total_ms, "calls": arr[i].calls,
                                   "launches": arr[i].launches} for i in range(n.value)}
