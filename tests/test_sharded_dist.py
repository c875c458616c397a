"""The token-sharded backward's host logic on CPU, with gloo ranks (world size
2 and 3): the token split, the gather of every rank's partials in rank order,
and the fixed-order combine that makes every rank's result the same bits.

Each rank computes its partials with the fp64 oracle on its own token slice
(the CUDA part of this path, smla_bwd_partial and smla_reduce_partials, is
tested on a GPU in test_gpu_sharded.py); the combine here is an fp32 sum in
rank order, the same order the library kernel uses.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from sparse_mla_attention_gb300.sharded import gather_in_rank_order, shard_bounds


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_in_order():
    for T in (0, 1, 7, 128, 1000):
        for world in (1, 2, 3, 8):
            bounds = [shard_bounds(T, world, r) for r in range(world)]
            assert bounds[0][0] == 0 and bounds[-1][1] == T
            assert all(bounds[r][1] == bounds[r + 1][0] for r in range(world - 1))
            sizes = [b - a for a, b in bounds]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)


def _case():
    from gpu_helpers import custom_inputs
    return custom_inputs(21, T=24, H=16, K=12, N=40, sink=True, mask_p=0.2)


def _partials(inp, t0, t1):
    """fp32 partials of tokens [t0, t1): dkv [N*512] then d_sink [H] (oracle)."""
    import oracle
    q = oracle.bf16_to_f64(inp["q"][t0:t1])
    kv = oracle.bf16_to_f64(inp["kv"])
    do = oracle.bf16_to_f64(inp["do"][t0:t1])
    topk = np.ascontiguousarray(inp["topk"][t0:t1])
    sink = inp["sink"].astype(np.float64)
    o_full, lse_full = oracle.fwd(oracle.bf16_to_f64(inp["q"]), kv, inp["topk"], sink, inp["scale"])
    o = o_full[t0:t1]
    lse = lse_full[t0:t1]
    ref = oracle.bwd(q, kv, do, o, lse, topk, sink, inp["scale"])
    return np.concatenate([ref["dkv"].reshape(-1), ref["dsink"]]).astype(np.float32)


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _case()
        T = inp["q"].shape[0]
        t0, t1 = shard_bounds(T, world, rank)
        local = torch.from_numpy(_partials(inp, t0, t1))
        parts = gather_in_rank_order(local)
        # every row is its rank's partial, in rank order
        mine = parts[rank].numpy()
        assert np.array_equal(mine, local.numpy())
        # the combine: fp32 additions in rank order
        acc = parts[0].numpy().copy()
        for r in range(1, world):
            acc = (acc + parts[r].numpy()).astype(np.float32)
        out[rank] = (parts.numpy().tobytes(), acc.tobytes())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gather_in_rank_order_and_ordered_combine_gloo(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    # every rank gathered the same partials and combined them into the same bits
    assert len({res[r][0] for r in range(world)}) == 1
    assert len({res[r][1] for r in range(world)}) == 1
    # the rows are the ranks' own slices, in rank order, and the combine is the
    # full backward's dkv and d_sink
    inp = _case()
    T = inp["q"].shape[0]
    parts = np.frombuffer(res[0][0], dtype=np.float32).reshape(world, -1)
    for r in range(world):
        t0, t1 = shard_bounds(T, world, r)
        assert np.array_equal(parts[r], _partials(inp, t0, t1))
    full = _partials(inp, 0, T)
    got = np.frombuffer(res[0][1], dtype=np.float32)
    np.testing.assert_allclose(got, full, rtol=1e-5, atol=1e-5 * np.max(np.abs(full)))
