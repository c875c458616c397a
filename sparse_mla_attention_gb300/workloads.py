"""Seeded synthetic inputs for the sparse MLA attention backward.

This module only draws random numbers and lays out index tables. It holds
none of the attention arithmetic: no scores, no softmax, no gradients. Both
the CUDA path and the CPU oracle read the arrays it returns; nothing here
depends on either of them.

The workloads stand in for the "realistic SWA(128)+pool top-k" inputs that
the aiter sparse-MLA backward page ("Sparse MLA training backward",
Performance section) times at T=4096, H=128, topk=512. That page publishes
no dataset or index table, so every tensor is drawn here:

* q, kv, dO ~ N(0, 1), rounded to bf16 (round to nearest even), returned as
  uint16 bit patterns;
* attn_sink ~ N(0, 1) fp32 per head (or absent);
* topk_indices int32 [T, topk]: each row lists the causal sliding-window
  rows ascending, then the pool picks ascending, then -1 padding.

Each tensor draws from its own child stream of ``numpy.random.SeedSequence``
so that changing one shape never perturbs another tensor.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

D_HEAD = 512  # the contract fixes the shared-KV width at 512


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and index recipe of one synthetic workload."""

    name: str
    T: int
    H: int
    topk: int
    num_kv: int
    window: int            # causal window length (rows t-window+1 .. t)
    pool_picks: int        # pool rows picked per token (0: no pool)
    pool_dist: str = "uniform"   # "uniform" or "zipf"
    zipf_s: float = 1.1
    mask_frac: float = 0.0       # fraction of all slots set to -1 at random
    sink: bool = True
    r_chunk: int = 0             # 0: ranks processed in one chunk
    D: int = D_HEAD

    @property
    def pool_rows(self) -> int:
        return self.num_kv - self.T

    def describe(self) -> str:
        return (f"T={self.T},H={self.H},D={self.D},topk={self.topk},"
                f"num_kv={self.num_kv},window={self.window},"
                f"pool_picks={self.pool_picks}({self.pool_dist}),"
                f"mask_frac={self.mask_frac},sink={self.sink},"
                f"r_chunk={self.r_chunk or self.topk}")


# The five workloads. "headline" is the one the aiter page times.
WORKLOADS = {
    "tiny": WorkloadSpec("tiny", T=128, H=16, topk=64, num_kv=128,
                         window=64, pool_picks=0),
    "t1024_h64": WorkloadSpec("t1024_h64", T=1024, H=64, topk=256, num_kv=1280,
                              window=128, pool_picks=128),
    "headline": WorkloadSpec("headline", T=4096, H=128, topk=512, num_kv=5120,
                             window=128, pool_picks=384),
    "headline_h64_chunked": WorkloadSpec("headline_h64_chunked", T=4096, H=64,
                                         topk=512, num_kv=5120, window=128,
                                         pool_picks=384, r_chunk=128),
    "t8192_zipf": WorkloadSpec("t8192_zipf", T=8192, H=128, topk=512,
                               num_kv=9216, window=128, pool_picks=384,
                               pool_dist="zipf", zipf_s=1.1, mask_frac=0.3,
                               sink=False),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest even); return the bit patterns.

    The inputs are finite normal samples, so the 32-bit carry never overflows.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_u.size, step):
        c = flat_u[i:i + step]
        flat_o[i:i + step] = (c + np.uint32(0x7FFF) + ((c >> 16) & np.uint32(1))) >> 16
    return out


_SLAB = 1 << 22


def _normal_bf16(seed_seq: np.random.SeedSequence, shape) -> np.ndarray:
    """N(0,1) samples rounded to bf16.

    The tensor is cut into fixed slabs of 2**22 values, each drawn from its own
    child stream of ``seed_seq``, so the values do not depend on how many
    threads fill them.
    """
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    nslab = (flat.size + _SLAB - 1) // _SLAB
    children = seed_seq.spawn(nslab)

    def fill(i: int) -> None:
        lo = i * _SLAB
        n = min(_SLAB, flat.size - lo)
        g = np.random.Generator(np.random.PCG64(children[i]))
        flat[lo:lo + n] = f32_to_bf16_bits(g.standard_normal(n, dtype=np.float32))

    if nslab == 1:
        fill(0)
    else:
        import concurrent.futures as cf
        import os
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nslab)))
    return out


def _pool_picks(rng: np.random.Generator, spec: WorkloadSpec) -> np.ndarray:
    """[T, pool_picks] distinct pool rows per token, ascending."""
    T, npool, k = spec.T, spec.pool_rows, spec.pool_picks
    if k == 0:
        return np.zeros((T, 0), dtype=np.int64)
    if k > npool:
        raise ValueError("more pool picks than pool rows")
    if spec.pool_dist == "uniform":
        keys = rng.random((T, npool))
    elif spec.pool_dist == "zipf":
        # Weighted draw without replacement by Gumbel-top-k: pool rank
        # k (1-based) has weight k**-s and maps to kv row T + k - 1.
        ranks = np.arange(1, npool + 1, dtype=np.float64)
        logw = -spec.zipf_s * np.log(ranks)
        gumbel = -np.log(-np.log(rng.random((T, npool)).clip(1e-300, 1.0)))
        keys = -(logw[None, :] + gumbel)      # smallest key = picked first
    else:
        raise ValueError(f"unknown pool distribution {spec.pool_dist!r}")
    picks = np.argpartition(keys, k - 1, axis=1)[:, :k]
    picks.sort(axis=1)
    return picks + spec.T


def make_topk(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    """Index table [T, topk] int32: window rows, pool picks, then -1."""
    T, K, W = spec.T, spec.topk, spec.window
    if W + spec.pool_picks > K:
        raise ValueError("window + pool picks exceed topk")
    out = np.full((T, K), -1, dtype=np.int64)
    t = np.arange(T)[:, None]
    w = np.arange(W)[None, :]
    win = t - (W - 1) + w                      # rows t-W+1 .. t, ascending
    nwin = np.minimum(np.arange(T) + 1, W)     # valid window rows per token
    # left-align the valid window rows, -1 fill behind them
    shift = W - nwin
    src = np.clip(w + shift[:, None], 0, W - 1)
    winrows = np.take_along_axis(win, src, axis=1)
    winrows[w >= nwin[:, None]] = -1
    pool = _pool_picks(rng, spec)
    P = pool.shape[1]
    # pack: window rows (valid ones), then pool picks, then -1
    for_t = np.concatenate([winrows, pool, np.full((T, K - W - P), -1)], axis=1)
    # compact away the -1 holes of short windows so the padding sits at the tail
    valid = for_t >= 0
    order = np.argsort(~valid, axis=1, kind="stable")
    out = np.take_along_axis(for_t, order, axis=1)
    if spec.mask_frac > 0:
        drop = rng.random((T, K)) < spec.mask_frac
        out[drop] = -1
    return out.astype(np.int32)


def make_inputs(spec: WorkloadSpec, seed: int = 0, with_do: bool = True) -> dict:
    """Draw every input of one workload.

    Returns a dict with ``q``, ``kv``, ``do`` (uint16 bf16 bit patterns),
    ``sink`` (float32 [H] or None), ``topk`` (int32 [T, topk]), ``scale``
    (float, 1/sqrt(D)) and ``r_chunk``.
    """
    ss_topk, ss_q, ss_kv, ss_do, ss_sink = np.random.SeedSequence(seed).spawn(5)
    T, H, D, N = spec.T, spec.H, spec.D, spec.num_kv
    topk = make_topk(spec, np.random.Generator(np.random.PCG64(ss_topk)))
    q = _normal_bf16(ss_q, (T, H, D))
    kv = _normal_bf16(ss_kv, (N, D))
    do = _normal_bf16(ss_do, (T, H, D)) if with_do else None
    r_sink = np.random.Generator(np.random.PCG64(ss_sink))
    sink: Optional[np.ndarray] = (
        r_sink.standard_normal(H, dtype=np.float32) if spec.sink else None)
    return {
        "spec": spec, "q": q, "kv": kv, "do": do, "sink": sink, "topk": topk,
        "scale": float(1.0 / np.sqrt(D)), "r_chunk": spec.r_chunk or spec.topk,
    }


def valid_ranks(topk: np.ndarray) -> int:
    """Number of (t, rank) slots that hold a row index (not -1)."""
    return int(np.count_nonzero(np.asarray(topk) >= 0))


def flops_valid(topk: np.ndarray, H: int, D: int = D_HEAD) -> float:
    """Backward FLOPs counting 5 GEMMs x 2 x D per valid (t, h, rank)."""
    return 5.0 * 2.0 * D * H * valid_ranks(topk)


def flops_nominal(T: int, H: int, topk: int, D: int = D_HEAD) -> float:
    """Backward FLOPs over all T*H*topk ranks, masked ones included.

    This is the count that reproduces the TFLOPS figures of the aiter page's
    Performance table (e.g. 3.380 ms -> 407 TFLOPS at T=4096 H=128 topk=512).
    """
    return 5.0 * 2.0 * D * H * float(T) * float(topk)
