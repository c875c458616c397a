"""The kernels' bounded waits, run out on purpose without faulting the GPU.

smla_selftest_wait_timeout launches one CTA that waits, through the same
wait-and-unwind code as the tensor-core kernels, on an mbarrier that nothing
arrives on, with a 1 ms limit. The wait must end by itself, the status word
must read SMLA_ERR_TIMEOUT, and the device must stay usable: a backward right
after it matches the oracle.
"""

import ctypes
import time

import pytest
import torch

import sparse_mla_attention_gb300 as smla
from sparse_mla_attention_gb300 import _lib
from gpu_helpers import Case, compare, custom_inputs, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    lib = _lib.load()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.smla_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), ws.numel(), 1000, stream)
    assert rc == _lib.SMLA_OK
    assert smla.device_status(ws) == _lib.SMLA_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0
    # argument checks happen on the host, before any launch
    assert lib.smla_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), ws.numel(), 0,
                                          stream) == _lib.SMLA_ERR_ARG
    assert lib.smla_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 16, 1000,
                                          stream) == _lib.SMLA_ERR_WORKSPACE
    host = torch.zeros(256, dtype=torch.uint8)
    assert lib.smla_selftest_wait_timeout(ctypes.c_void_p(host.data_ptr()), 256, 1000,
                                          stream) == _lib.SMLA_ERR_DEVICE
    # the context is still usable: a backward right after is correct
    c = Case(custom_inputs(5, T=40, H=32, K=48, N=90, sink=True))
    dq, dkv, ds = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
    ref = c.ref_full()
    compare("dq", to_f64(dq), ref["dq"])
    compare("dkv", to_f64(dkv), ref["dkv"])
    compare("d_sink", to_f64(ds), ref["dsink"])
