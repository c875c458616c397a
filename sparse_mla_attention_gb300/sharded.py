"""Token-sharded backward over several GPUs (one process per GPU).

Each rank holds a contiguous slice of the tokens (q, dO, O, lse, topk rows)
and the full kv (and sink). It runs ``smla_bwd_partial`` on its slice: dq of
its tokens is final; the kv and sink gradients are fp32 partial sums over its
tokens. The partials of all ranks are then gathered (the collective only
moves data) and added in rank order by ``smla_reduce_partials``, which rounds
dkv to bf16 once. Every rank ends with the same dkv and d_sink bits: the
RL-Kernel page's "Algorithmic arrangements" item 5, a fixed-order reduction
with the communication library used as transport, never as the reducer.
"""

from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

from . import api


def shard_bounds(T: int, world: int, rank: int) -> Tuple[int, int]:
    """Token range [t0, t1) of `rank` when T tokens are split into `world`
    contiguous slices whose sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("need world >= 1, 0 <= rank < world and T >= 0")
    base, extra = divmod(T, world)
    t0 = rank * base + min(rank, extra)
    return t0, t0 + base + (1 if rank < extra else 0)


def gather_in_rank_order(local: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' 1-D tensors of equal length stacked as [world, n], row r from
    rank r (all_gather_into_tensor: data movement only)."""
    if local.dim() != 1:
        raise ValueError("local must be 1-D")
    world = dist.get_world_size(group)
    out = torch.empty(world * local.numel(), dtype=local.dtype, device=local.device)
    dist.all_gather_into_tensor(out, local.contiguous(), group=group)
    return out.view(world, local.numel())


def sparse_mla_bwd_sharded(q: torch.Tensor, kv: torch.Tensor, do: torch.Tensor, o: torch.Tensor,
                           lse: torch.Tensor, topk: torch.Tensor, sink: Optional[torch.Tensor] = None,
                           scale: Optional[float] = None, r_chunk: Optional[int] = None,
                           group=None, workspace: Optional[api.Workspace] = None):
    """This rank's part of a token-sharded backward.

    q, do, o, lse, topk: this rank's token slice (see shard_bounds); kv, sink:
    the full tensors, the same on every rank. Returns (dq of the slice [T_r,H,512]
    bf16, dkv [num_kv,512] bf16, d_sink [H] fp32 or None); dkv and d_sink are
    identical on every rank of the group.
    """
    dq, dkv_p, ds_p = api.sparse_mla_bwd_partial(q, kv, do, o, lse, topk, sink, scale=scale,
                                                 r_chunk=r_chunk, workspace=workspace)
    n_kv = dkv_p.numel()
    local = dkv_p.reshape(-1) if ds_p is None else torch.cat([dkv_p.reshape(-1), ds_p])
    parts = gather_in_rank_order(local, group)
    s_bf16, s_f32 = api.reduce_partials(parts, want_bf16=True, want_f32=ds_p is not None)
    dkv = s_bf16[:n_kv].view(kv.shape)
    d_sink = None if ds_p is None else s_f32[n_kv:].clone()
    return dq, dkv, d_sink
