"""Token-sharded backward on one GPU: the shards run one after the other
through smla_bwd_partial, their fp32 partials are added in rank order by
smla_reduce_partials, and the result is checked against the fp64 oracle of
the whole problem (and is the same bits on every repeat)."""

import os
import socket

import numpy as np
import pytest
import torch

import sparse_mla_attention_gb300 as smla
from sparse_mla_attention_gb300 import workloads as W
from sparse_mla_attention_gb300.sharded import shard_bounds
from gpu_helpers import Case, compare, custom_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def t1024():
    return Case(W.make_inputs(W.WORKLOADS["t1024_h64"]))


def test_reduce_partials_adds_in_rank_order():
    # fp32 addition is not associative: (1e8 + 1) - 1e8 = 0 but 1e8 + (1 - 1e8) = 1
    n = 1024
    rng = np.random.default_rng(3)
    parts = rng.standard_normal((3, n)).astype(np.float32) * np.float32(1e3)
    parts[0, :4] = [1e8, -1e8, 3.0, 2.0 ** 24]
    parts[1, :4] = [1.0, 1.0, 1e8, 1.0]
    parts[2, :4] = [-1e8, 1e8, -1e8, 1.0]
    want = ((parts[0] + parts[1]).astype(np.float32) + parts[2]).astype(np.float32)
    dev = torch.from_numpy(parts).cuda()
    got_b, got_f = smla.reduce_partials(dev, want_bf16=True, want_f32=True)
    assert np.array_equal(got_f.cpu().numpy(), want)
    assert torch.equal(got_b, torch.from_numpy(want).cuda().to(torch.bfloat16))
    assert got_f.cpu().numpy()[0] == 0.0 and got_f.cpu().numpy()[1] == 0.0


def _slices(c, t0, t1):
    return (c.q[t0:t1], c.do[t0:t1], c.o[t0:t1], c.lse[t0:t1], c.topk[t0:t1])


def _sharded(c, world, r_chunk=None):
    dqs, dkvs, dss = [], [], []
    for r in range(world):
        t0, t1 = shard_bounds(c.T, world, r)
        q, do, o, lse, topk = _slices(c, t0, t1)
        dq, dkv_p, ds_p = smla.sparse_mla_bwd_partial(q, c.kv, do, o, lse, topk, c.sink,
                                                      r_chunk=r_chunk)
        dqs.append(dq)
        dkvs.append(dkv_p.reshape(-1))
        dss.append(ds_p)
    dkv_b, _ = smla.reduce_partials(torch.stack(dkvs), want_bf16=True)
    _, ds_f = smla.reduce_partials(torch.stack(dss), want_bf16=False, want_f32=True)
    return torch.cat(dqs), dkv_b.view(c.kv.shape), ds_f


@pytest.mark.parametrize("world,r_chunk", [(2, None), (3, 128)])
def test_two_and_three_shards_match_the_oracle(t1024, world, r_chunk):
    c = t1024
    dq, dkv, ds = _sharded(c, world, r_chunk)
    ref = c.ref_full()
    compare("dq (sharded)", to_f64(dq), ref["dq"])
    compare("dkv (sharded)", to_f64(dkv), ref["dkv"])
    compare("d_sink (sharded)", to_f64(ds), ref["dsink"])
    # the same bits on a repeat
    dq2, dkv2, ds2 = _sharded(c, world, r_chunk)
    assert torch.equal(dq, dq2) and torch.equal(dkv, dkv2) and torch.equal(ds, ds2)
    # and close to the one-GPU backward (the summation order of dkv differs)
    dq1, dkv1, ds1 = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink,
                                         r_chunk=r_chunk)
    # dq of a token depends on that token alone: the same bits as unsharded
    assert torch.equal(dq, dq1)
    compare("dkv vs unsharded", to_f64(dkv), to_f64(dkv1), cos_min=0.99999, rel=1e-2)


def test_partial_of_a_single_shard_is_the_unrounded_dkv(t1024):
    c = t1024
    _, dkv_p, ds_p = smla.sparse_mla_bwd_partial(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
    _, dkv, ds = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
    assert dkv_p.dtype == torch.float32
    # one shard: the partial rounded once is the backward's dkv, and d_sink is the same
    assert torch.equal(dkv_p.to(torch.bfloat16), dkv)
    assert torch.equal(ds_p, ds)


def test_partial_empty_shard_is_zero():
    H, N = 16, 10
    q = torch.zeros((0, H, 512), dtype=torch.bfloat16, device="cuda")
    kv = torch.randn((N, 512), device="cuda").bfloat16()
    topk = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    lse = torch.zeros((0, H), dtype=torch.float32, device="cuda")
    sink = torch.randn(H, device="cuda")
    dq, dkv_p, ds_p = smla.sparse_mla_bwd_partial(q, kv, q, q, lse, topk, sink)
    assert dq.numel() == 0 and torch.all(dkv_p == 0) and torch.all(ds_p == 0)


def test_sharded_helper_world_of_one(t1024):
    # the torch.distributed path end to end on one GPU (a one-rank NCCL group)
    import torch.distributed as dist
    from sparse_mla_attention_gb300.sharded import sparse_mla_bwd_sharded
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        c = t1024
        dq, dkv, ds = sparse_mla_bwd_sharded(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
        _, dkv_p, ds_p = smla.sparse_mla_bwd_partial(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink)
        assert torch.equal(dkv, dkv_p.to(torch.bfloat16)) and torch.equal(ds, ds_p)
    finally:
        dist.destroy_process_group()
