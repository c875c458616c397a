"""fp64 CPU oracle for sparse MLA attention -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product package never does, and
this package never imports the product package: the two share nothing but
the seeded inputs of ``sparse_mla_attention_gb300.workloads``.

The arithmetic lives in ``smla_oracle.c`` (plain C, double accumulation,
OpenMP over independent outputs). This module builds it with gcc, loads it
with ctypes and converts bf16 / fp32 bit patterns to double exactly.

Every function follows the aiter page "[WIP][TRITON][GLUON][GFX950][DSV4]
Sparse MLA training backward" (sections "Contract" and "Structure"); the
C file states each definition next to its code.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smla_oracle.c")
_LIB = os.path.join(_HERE, "libsmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no CUDA involved)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.smla_oracle_threads.restype = ctypes.c_int
            lib.smla_oracle_fwd.argtypes = [i64] * 5 + [dp, dp, ip, dp, ctypes.c_double, dp, dp]
            lib.smla_oracle_bwd.argtypes = ([i64] * 5 + [dp] * 5 + [ip, dp, ctypes.c_double]
                                            + [dp] * 4)
            lib.smla_oracle_csr.argtypes = [ip] + [i64] * 5 + [ip, ip]
            lib.smla_oracle_dkv_rows.argtypes = ([i64] * 5 + [dp] * 5 + [ip, ctypes.c_double,
                                                 i64, i64, ip, ip, ip, i64, dp])
            lib.smla_oracle_dq_tokens.argtypes = ([i64] * 5 + [dp] * 5 + [ip, ctypes.c_double,
                                                  ip, i64, dp])
            lib.smla_oracle_dsink.argtypes = [i64] * 3 + [dp] * 5
            for f in ("smla_oracle_fwd", "smla_oracle_bwd", "smla_oracle_csr",
                      "smla_oracle_dkv_rows", "smla_oracle_dq_tokens", "smla_oracle_dsink"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().smla_oracle_threads())


# ---------------------------------------------------------------- conversions
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (via fp32, nearest even).

    Used only to turn the oracle's fp64 forward output O into the bf16 input
    the backward takes; any faithful rounding gives a valid input.
    """
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# ------------------------------------------------------------------- the math
def fwd(q, kv, topk, sink, scale):
    """Forward: returns (O [T,H,D] float64, lse [T,H] float64).

    q [T,H,D], kv [N,D] (float64), topk [T,K] int32, sink [H] or None.
    """
    q, kv, topk = _f64(q), _f64(kv), _i32(topk)
    T, H, D = q.shape
    N, K = kv.shape[0], topk.shape[1]
    s = None if sink is None else _f64(sink)
    o = np.empty((T, H, D)); lse = np.empty((T, H))
    _check(_load().smla_oracle_fwd(T, H, D, K, N, _p(q), _p(kv), _p(topk), _p(s),
                                   float(scale), _p(o), _p(lse)), "fwd")
    return o, lse


def bwd(q, kv, do, o, lse, topk, sink, scale, want=("dq", "dkv", "dsink", "delta")):
    """Full backward (small problems): dict with dq, dkv, dsink, delta (float64)."""
    q, kv, do, o, lse, topk = _f64(q), _f64(kv), _f64(do), _f64(o), _f64(lse), _i32(topk)
    T, H, D = q.shape
    N, K = kv.shape[0], topk.shape[1]
    s = None if sink is None else _f64(sink)
    out = {
        "dq": np.empty((T, H, D)) if "dq" in want else None,
        "dkv": np.empty((N, D)) if "dkv" in want else None,
        "dsink": np.empty(H) if ("dsink" in want and s is not None) else None,
        "delta": np.empty((T, H)) if "delta" in want else None,
    }
    _check(_load().smla_oracle_bwd(T, H, D, K, N, _p(q), _p(kv), _p(do), _p(o), _p(lse),
                                   _p(topk), _p(s), float(scale), _p(out["dq"]),
                                   _p(out["dkv"]), _p(out["dsink"]), _p(out["delta"])),
           "bwd")
    return out


def csr(topk, num_kv, r0=0, r_len=None):
    """Inverted top-k CSR over ranks [r0, r0+r_len): (row_ptr [N+1], col [nnz]) int32."""
    topk = _i32(topk)
    T, Kw = topk.shape
    R = Kw - r0 if r_len is None else r_len
    row_ptr = np.empty(num_kv + 1, dtype=np.int32)
    col = np.empty(T * R, dtype=np.int32)
    _check(_load().smla_oracle_csr(_p(topk), T, Kw, r0, R, num_kv, _p(row_ptr), _p(col)),
           "csr")
    return row_ptr, col[: int(row_ptr[-1])].copy()


def dkv_rows(q, kv, do, o, lse, topk, scale, rows: Sequence[int], r_chunk=None):
    """dkv for the given kv rows by the CSR-gather form, chunks summed in order."""
    q, kv, do, o, lse, topk = _f64(q), _f64(kv), _f64(do), _f64(o), _f64(lse), _i32(topk)
    T, H, D = q.shape
    N, K = kv.shape[0], topk.shape[1]
    R = r_chunk or K
    rows_a = np.ascontiguousarray(rows, dtype=np.int64)
    total = np.zeros((rows_a.size, D))
    for r0 in range(0, K, R):
        row_ptr, col = csr(topk, N, r0, R)
        col_full = np.ascontiguousarray(col, dtype=np.int32)
        part = np.empty((rows_a.size, D))
        _check(_load().smla_oracle_dkv_rows(T, H, D, K, N, _p(q), _p(kv), _p(do), _p(o),
                                            _p(lse), _p(topk), float(scale), r0, R,
                                            _p(row_ptr), _p(col_full), _p(rows_a),
                                            rows_a.size, _p(part)), "dkv_rows")
        total += part
    return total


def dq_tokens(q, kv, do, o, lse, topk, scale, tokens: Sequence[int]):
    """dq for the given tokens: [len(tokens), H, D] float64."""
    q, kv, do, o, lse, topk = _f64(q), _f64(kv), _f64(do), _f64(o), _f64(lse), _i32(topk)
    T, H, D = q.shape
    N, K = kv.shape[0], topk.shape[1]
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    out = np.empty((tok.size, H, D))
    _check(_load().smla_oracle_dq_tokens(T, H, D, K, N, _p(q), _p(kv), _p(do), _p(o),
                                         _p(lse), _p(topk), float(scale), _p(tok),
                                         tok.size, _p(out)), "dq_tokens")
    return out


def dsink(do, o, lse, sink):
    """(d_sink [H], delta [T,H]) float64."""
    do, o, lse, s = _f64(do), _f64(o), _f64(lse), _f64(sink)
    T, H, D = do.shape
    ds = np.empty(H); delta = np.empty((T, H))
    _check(_load().smla_oracle_dsink(T, H, D, _p(do), _p(o), _p(lse), _p(s), _p(ds),
                                     _p(delta)), "dsink")
    return ds, delta


def fwd_inputs(inp: dict):
    """Oracle forward on a workload dict; returns (o_bf16_bits, lse_f32, o_f64, lse_f64).

    The backward's O input is the fp64 O rounded to bf16 and its lse input is
    the fp64 lse rounded to fp32, as a bf16 forward would hand them over.
    """
    q = bf16_to_f64(inp["q"]); kv = bf16_to_f64(inp["kv"])
    o, lse = fwd(q, kv, inp["topk"], inp["sink"], inp["scale"])
    return f64_to_bf16(o), lse.astype(np.float32), o, lse
