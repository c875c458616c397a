"""GPU tests of smla_bwd_host, the backward with host inputs and outputs.

Its results must equal those of smla_bwd on the same inputs bit for bit (the
token-chunked schedule runs the same kernels on the same data), and match
the fp64 oracle; pinned and pageable host memory, rank chunking, several
token chunks and T == 0 are covered.
"""

import pytest
import torch

import oracle
import sparse_mla_attention_gb300 as smla
from sparse_mla_attention_gb300 import workloads as W
from gpu_helpers import Case, compare, custom_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mla_attention_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _host(c: Case, pin: bool):
    f = (lambda t: t.cpu().pin_memory()) if pin else (lambda t: t.cpu())
    return [f(t) if t is not None else None for t in (c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)]


def _same(dev_out, host_out):
    for a, b in zip(dev_out, host_out):
        if a is None:
            assert b is None
        else:
            assert torch.equal(a.cpu(), b), "host-buffer results differ from the device path"


@pytest.mark.parametrize("pin,r_chunk", [(True, None), (False, None), (True, 128)])
def test_bwd_host_equals_device_path(pin, r_chunk):
    # T = 1024: two token chunks of 512
    c = Case(W.make_inputs(W.WORKLOADS["t1024_h64"]))
    dev = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, scale=c.scale,
                              r_chunk=r_chunk)
    q, kv, do, o, lse, topk, sink = _host(c, pin)
    host = smla.sparse_mla_bwd_host(q, kv, do, o, lse, topk, sink, scale=c.scale, r_chunk=r_chunk)
    _same(dev, host)
    if r_chunk is None and pin:
        ref = c.ref_full()
        compare("dq (host path)", to_f64(host[0]), ref["dq"])
        compare("dkv (host path)", to_f64(host[1]), ref["dkv"])
        compare("d_sink (host path)", to_f64(host[2]), ref["dsink"])


def test_bwd_host_ragged_token_chunks_no_sink():
    # T = 1300: three token chunks (433 / 433 / 434 tokens), topk not a multiple of 128
    c = Case(custom_inputs(77, T=1300, H=32, K=200, N=1400, sink=False,
                           all_masked_rows=(5,), r_chunk=0))
    dev = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, None, scale=c.scale)
    q, kv, do, o, lse, topk, _ = _host(c, True)
    host = smla.sparse_mla_bwd_host(q, kv, do, o, lse, topk, None, scale=c.scale)
    _same(dev, host)
    assert host[2] is None


def test_bwd_host_empty_T():
    H, N = 16, 10
    q = torch.zeros((0, H, 512), dtype=torch.bfloat16)
    kv = torch.randn((N, 512)).bfloat16()
    topk = torch.zeros((0, 4), dtype=torch.int32)
    lse = torch.zeros((0, H), dtype=torch.float32)
    sink = torch.randn(H)
    dq, dkv, ds = smla.sparse_mla_bwd_host(q, kv, q, q, lse, topk, sink)
    assert dq.numel() == 0 and torch.all(dkv == 0) and torch.all(ds == 0)


def test_bwd_host_rejects_device_tensors():
    c = Case(W.make_inputs(W.WORKLOADS["tiny"]))
    with pytest.raises(ValueError):
        smla.sparse_mla_bwd_host(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
