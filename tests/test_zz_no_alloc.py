"""The allocation-free d_sink entry point (smla_dsink_static).

Some callers cannot allocate device memory (another allocator owns it all,
or allocating is not allowed where they run), so they cannot pass smla_bwd a
workspace. smla_dsink_static serves them with its scratch in a static device
array. This test calls it through the C ABI twice in a row and checks both
results against the fp64 oracle (at the parity bar) and, bit for bit,
against the d_sink of smla_bwd on the same inputs (same kernels).

The file name sorts last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import Case, compare, to_f64

pytestmark = pytest.mark.gpu


def _case():
    from sparse_mla_attention_gb300 import workloads as W
    # O and lse come from the oracle's forward (never from the CUDA path)
    return Case(W.make_inputs(W.WORKLOADS["t1024_h64"]))


def _call_static(lib, do, o, lse, sink, d_sink, T, H):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.smla_dsink_static(p(do), p(o), p(lse), p(sink), p(d_sink), T, H, stream)


def test_static_dsink_matches_oracle_and_bwd_twice():
    from sparse_mla_attention_gb300 import _lib, build
    build.build()
    import sparse_mla_attention_gb300 as smla
    lib = _lib.load()
    c = _case()
    T, H = c.T, c.H
    _, _, from_bwd = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
    ref = c.ref_dsink()
    outs = []
    for _ in range(2):
        d_sink = torch.full((H,), float("nan"), device="cuda")
        assert _call_static(lib, c.do, c.o, c.lse, c.sink, d_sink, T, H) == _lib.SMLA_OK
        torch.cuda.synchronize()
        outs.append(d_sink)
    for d_sink in outs:
        # against the fp64 oracle, at the bar of every parity test
        compare("d_sink (static)", to_f64(d_sink), ref)
        # the same kernels on the same inputs as smla_bwd's d_sink: equal bit for bit
        assert torch.equal(d_sink, from_bwd)
    assert torch.equal(outs[0], outs[1])


def test_static_dsink_rejects_sizes_over_the_limit():
    from sparse_mla_attention_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    H = 128
    T = (1 << 20) // H + 1           # one token past the 2^20-entry scratch
    small = torch.zeros(16, device="cuda")
    d_sink = torch.zeros(H, device="cuda")
    rc = _call_static(lib, small, small, small, small, d_sink, T, H)
    assert rc == _lib.SMLA_ERR_SHAPE
