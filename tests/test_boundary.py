"""Host-side tests of the C ABI (no GPU needed).

Validation in libsmla.so happens before any CUDA call, so calls with bad
arguments return their error code on a machine without a GPU; the fake
device pointers below are never dereferenced.
"""

import ctypes
import os
import re

import pytest

from sparse_mla_attention_gb300 import _lib, build as smla_build
from sparse_mla_attention_gb300._lib import SmlaDims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    smla_build.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smla_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(names) == set(_lib.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert lib.smla_version() == 100
    for code in range(0, 16):
        s = lib.smla_status_string(code)
        assert s and s != b"unknown status code"
    assert lib.smla_status_string(999) == b"unknown status code"


BASE = dict(T=64, H=16, D=512, topk=32, num_kv=80, r_chunk=0, scale=0.0)
# Fake, 16-byte aligned, non-overlapping "device" addresses (never touched).
GB = 1 << 30


def _addrs():
    return {k: ctypes.c_void_p((i + 1) * GB) for i, k in enumerate(
        ["q", "kv", "do", "o", "lse", "topk", "sink", "dq", "dkv", "dsink", "ws"])}


def _bwd(lib, dims, a, ws_bytes=None):
    if ws_bytes is None:
        n = ctypes.c_size_t()
        rc = lib.smla_workspace_size(_lib.SMLA_OP_BWD, ctypes.byref(dims), ctypes.byref(n))
        if rc:
            return rc
        ws_bytes = n.value
    return lib.smla_bwd(a["q"], a["kv"], a["do"], a["o"], a["lse"], a["topk"], a["sink"],
                        a["dq"], a["dkv"], a["dsink"], ctypes.byref(dims), a["ws"], ws_bytes, None)


@pytest.mark.parametrize("change,code", [
    (dict(D=256), _lib.SMLA_ERR_D512),
    (dict(num_kv=63), _lib.SMLA_ERR_NUM_KV_LT_T),
    (dict(r_chunk=5), _lib.SMLA_ERR_RCHUNK),
    (dict(r_chunk=64), _lib.SMLA_ERR_RCHUNK),
    (dict(H=24), _lib.SMLA_ERR_SHAPE),
    (dict(H=256), _lib.SMLA_ERR_SHAPE),
    (dict(topk=0), _lib.SMLA_ERR_SHAPE),
    (dict(T=-1), _lib.SMLA_ERR_SHAPE),
    (dict(scale=float("nan")), _lib.SMLA_ERR_ARG),
    (dict(scale=-1.0), _lib.SMLA_ERR_ARG),
])
def test_bwd_rejects_bad_dims(lib, change, code):
    dims = SmlaDims(**{**BASE, **change})
    assert _bwd(lib, dims, _addrs()) == code


def test_bwd_rejects_bad_pointers(lib):
    dims = SmlaDims(**BASE)
    a = _addrs(); a["q"] = None
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_NULL
    a = _addrs(); a["ws"] = None
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_NULL
    a = _addrs(); a["dsink"] = None                       # sink given, d_sink missing
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_SINK
    a = _addrs(); a["sink"] = None                        # d_sink without sink
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_SINK
    a = _addrs(); a["kv"] = ctypes.c_void_p(2 * GB + 8)
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_ALIGN
    a = _addrs(); a["dq"] = a["q"]                        # output over an input
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_OVERLAP
    a = _addrs(); a["dkv"] = ctypes.c_void_p(a["dq"].value + 4096)   # two outputs overlap
    assert _bwd(lib, dims, a) == _lib.SMLA_ERR_OVERLAP
    a = _addrs()
    assert _bwd(lib, dims, a, ws_bytes=1024) == _lib.SMLA_ERR_WORKSPACE


def test_valid_call_reaches_the_device_check(lib):
    """With every argument valid the only remaining check is the device's."""
    import torch
    dims = SmlaDims(**BASE)
    rc = _bwd(lib, dims, _addrs())
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the device check is covered by the GPU tests")
    assert rc in (_lib.SMLA_ERR_CUDA, _lib.SMLA_ERR_ARCH)


def test_workspace_size_grows_with_chunks(lib):
    def ws(**kw):
        d = SmlaDims(**{**BASE, **kw})
        n = ctypes.c_size_t()
        assert lib.smla_workspace_size(_lib.SMLA_OP_BWD, ctypes.byref(d), ctypes.byref(n)) == 0
        return n.value
    full = ws(T=4096, H=128, topk=512, num_kv=5120)
    chunked = ws(T=4096, H=128, topk=512, num_kv=5120, r_chunk=128)
    # the [T, R, 512] bf16 intermediate dominates: 2 GiB unchunked at this shape
    assert full > 2 * (1 << 30) > chunked
    n = ctypes.c_size_t()
    d = SmlaDims(**BASE)
    assert lib.smla_workspace_size(_lib.SMLA_OP_FWD, ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value >= 4
    assert lib.smla_workspace_size(7, ctypes.byref(d), ctypes.byref(n)) == _lib.SMLA_ERR_ARG


def test_chunks_of_128_ranks_need_no_dq_accumulator(lib):
    def ws(**kw):
        d = SmlaDims(**{**BASE, "T": 4096, "H": 128, "topk": 512, "num_kv": 5120, **kw})
        n = ctypes.c_size_t()
        assert lib.smla_workspace_size(_lib.SMLA_OP_BWD, ctypes.byref(d), ctypes.byref(n)) == 0
        return n.value
    acc = 4096 * 128 * 512 * 4          # the fp32 dq accumulator of per-chunk dq: 1 GiB
    # r_chunk = 64 keeps a per-chunk dS^T stash and the fp32 dq accumulator; r_chunk = 128
    # (a multiple of 128) keeps one stash over all ranks and runs dq once, without it
    assert ws(r_chunk=64) > acc
    assert ws(r_chunk=128) < ws(r_chunk=64)


def test_csr_build_validation(lib):
    a = _addrs()
    big = ctypes.c_size_t(1 << 40).value
    f = lib.smla_csr_build
    assert f(None, 4, 8, 0, 8, 10, a["dq"], a["dkv"], a["ws"], big, None) == _lib.SMLA_ERR_NULL
    assert f(a["topk"], 4, 8, 4, 5, 10, a["dq"], a["dkv"], a["ws"], big, None) == _lib.SMLA_ERR_SHAPE
    assert f(a["topk"], 4, 8, 0, 8, 0, a["dq"], a["dkv"], a["ws"], big, None) == _lib.SMLA_ERR_SHAPE
    assert f(a["topk"], 4, 8, 0, 8, 10, a["dq"], a["dkv"], a["ws"], 16, None) == _lib.SMLA_ERR_WORKSPACE
    assert f(a["topk"], 4, 8, 0, 8, 10, a["topk"], a["dkv"], a["ws"], big, None) == _lib.SMLA_ERR_OVERLAP
    odd = ctypes.c_void_p(a["dq"].value + 4)
    assert f(a["topk"], 4, 8, 0, 8, 10, odd, a["dkv"], a["ws"], big, None) == _lib.SMLA_ERR_ALIGN


def test_fwd_validation(lib):
    a = _addrs()
    d = SmlaDims(**BASE)
    f = lib.smla_fwd
    assert f(a["q"], a["kv"], a["topk"], a["sink"], a["o"], a["lse"], ctypes.byref(d),
             a["ws"], 16, None) == _lib.SMLA_ERR_WORKSPACE
    assert f(a["q"], a["kv"], a["topk"], a["sink"], a["q"], a["lse"], ctypes.byref(d),
             a["ws"], 4096, None) == _lib.SMLA_ERR_OVERLAP
    d2 = SmlaDims(**{**BASE, "D": 128})
    assert f(a["q"], a["kv"], a["topk"], a["sink"], a["o"], a["lse"], ctypes.byref(d2),
             a["ws"], 4096, None) == _lib.SMLA_ERR_D512


def _bwd_host(lib, dims, a, ws_bytes=None):
    if ws_bytes is None:
        n = ctypes.c_size_t()
        rc = lib.smla_workspace_size(_lib.SMLA_OP_BWD_HOST, ctypes.byref(dims), ctypes.byref(n))
        if rc:
            return rc
        ws_bytes = n.value
    return lib.smla_bwd_host(a["q"], a["kv"], a["do"], a["o"], a["lse"], a["topk"], a["sink"],
                             a["dq"], a["dkv"], a["dsink"], ctypes.byref(dims), a["ws"], ws_bytes,
                             None)


def test_bwd_host_workspace_holds_device_copies(lib):
    d = SmlaDims(**{**BASE, "T": 4096, "H": 128, "topk": 512, "num_kv": 5120})
    n_dev, n_host = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.smla_workspace_size(_lib.SMLA_OP_BWD, ctypes.byref(d), ctypes.byref(n_dev)) == 0
    assert lib.smla_workspace_size(_lib.SMLA_OP_BWD_HOST, ctypes.byref(d), ctypes.byref(n_host)) == 0
    # q, dO, o and dq (4 x 512 MiB) plus kv, dkv, lse, topk and sink live in the workspace
    copies = 4 * 4096 * 128 * 512 * 2 + 2 * 5120 * 512 * 2 + 4096 * 128 * 4 + 4096 * 512 * 4
    assert n_host.value >= n_dev.value + copies


def test_bwd_host_validation(lib):
    dims = SmlaDims(**BASE)
    a = _addrs(); a["q"] = None
    assert _bwd_host(lib, dims, a) == _lib.SMLA_ERR_NULL
    a = _addrs(); a["dsink"] = None
    assert _bwd_host(lib, dims, a) == _lib.SMLA_ERR_SINK
    a = _addrs(); a["ws"] = ctypes.c_void_p(a["ws"].value + 8)
    assert _bwd_host(lib, dims, a) == _lib.SMLA_ERR_ALIGN
    a = _addrs(); a["dq"] = a["o"]
    assert _bwd_host(lib, dims, a) == _lib.SMLA_ERR_OVERLAP
    a = _addrs()
    assert _bwd_host(lib, dims, a, ws_bytes=4096) == _lib.SMLA_ERR_WORKSPACE
    assert _bwd_host(lib, SmlaDims(**{**BASE, "D": 128}), _addrs()) == _lib.SMLA_ERR_D512
    # host pointers need no 16-byte alignment: with a valid call the only check
    # left is the device's (the fake pointers must never reach a real copy)
    import torch
    if torch.cuda.is_available():
        return
    a = _addrs(); a["lse"] = ctypes.c_void_p(a["lse"].value + 4)
    assert _bwd_host(lib, dims, a) in (_lib.SMLA_ERR_CUDA, _lib.SMLA_ERR_ARCH)


def test_missing_library_fails_loudly():
    # no fallback: loading a library that is not there raises (fresh process, nothing cached)
    import subprocess
    import sys
    code = ("from sparse_mla_attention_gb300 import _lib\n"
            "_lib.load('/nonexistent/libsmla.so')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode != 0 and "not found" in r.stderr


def test_python_api_refuses_cpu_tensors():
    # the product path has no CPU fallback: host tensors are rejected before any call
    import torch
    import sparse_mla_attention_gb300 as smla
    T, H, K, N = 4, 16, 8, 10
    q = torch.zeros((T, H, 512), dtype=torch.bfloat16)
    kv = torch.zeros((N, 512), dtype=torch.bfloat16)
    topk = torch.zeros((T, K), dtype=torch.int32)
    lse = torch.zeros((T, H), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        smla.sparse_mla_fwd(q, kv, topk)
    with pytest.raises(ValueError, match="CUDA tensor"):
        smla.sparse_mla_bwd(q, kv, q, q, lse, topk)
