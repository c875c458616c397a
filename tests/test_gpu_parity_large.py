"""GPU parity at the full workload sizes, in the launch configuration bench.py
times (same shapes, same rank chunking), on outputs the fp64 oracle can
compute one by one:

* dq for at least 256 sampled tokens (the first and last tokens, the end of
  the short windows, and seeded random tokens);
* dkv for at least 64 sampled kv rows (window rows, pool rows, rows no token
  selects, and the rows with the most contributors -- the hottest Zipf rows in
  the skewed workload), each computed by the oracle from its full
  contributor list;
* all of d_sink;
plus bitwise run-to-run determinism of dq, dkv and d_sink; and the forward
(O and lse) on every token against the oracle's forward.

O and lse, the backward's inputs, come from the oracle's forward over all
tokens (never from the CUDA path).
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_gb300 as smla
from sparse_mla_attention_gb300 import workloads as W
from gpu_helpers import Case, compare, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mla_attention_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _sample_tokens(T, rng, n=256):
    # at least 256 tokens: the first and last tokens, the end of the short
    # windows, and seeded random tokens
    fixed = [0, 1, 2, 63, 126, 127, 128, T // 2, T - 2, T - 1]
    toks = set(fixed)
    for t in rng.permutation(T):
        if len(toks) >= n:
            break
        toks.add(int(t))
    return np.array(sorted(toks), dtype=np.int64)


def _sample_rows(topk, N, T, rng, n=64):
    # at least 64 kv rows: the hottest rows, window rows, pool rows, rows no
    # token selects, and the first / last rows
    counts = np.bincount(topk[topk >= 0], minlength=N)
    hottest = np.argsort(-counts, kind="stable")[:16]
    window = rng.choice(T, size=20, replace=False)
    pool = T + rng.choice(N - T, size=24, replace=False) if N > T else np.array([], np.int64)
    unused = np.flatnonzero(counts == 0)[:2]
    fixed = [0, T - 1, N - 1]
    rows = set(np.concatenate([hottest, window, pool, unused, fixed]).astype(np.int64).tolist())
    for j in rng.permutation(N):
        if len(rows) >= n:
            break
        rows.add(int(j))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.fixture(scope="module", params=["headline", "headline_h64_chunked", "t8192_zipf"])
def big(request):
    # module scope with parameters: pytest runs every test of one workload
    # before building the next, so one set of oracle arrays is alive at a time
    spec = W.WORKLOADS[request.param]
    inp = W.make_inputs(spec)
    return request.param, spec, inp, Case(inp)


def test_full_size_sampled_parity_and_determinism(big):
    name, spec, inp, c = big
    r_chunk = spec.r_chunk or None
    ws = smla.Workspace()
    out1 = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, scale=c.scale,
                               r_chunk=r_chunk, workspace=ws)
    out2 = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, scale=c.scale,
                               r_chunk=r_chunk, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(out1, out2):
        if a is not None:
            assert torch.equal(a, b), "run-to-run results differ"
    dq, dkv, dsink = out1

    rng = np.random.default_rng(123)
    toks = _sample_tokens(spec.T, rng)
    ref_dq = c.ref_dq(toks)
    compare(f"{name} dq[sampled tokens]", to_f64(dq[torch.from_numpy(toks).cuda()]), ref_dq)

    rows = _sample_rows(inp["topk"], spec.num_kv, spec.T, rng)
    ref_dkv = oracle.dkv_rows(c.q64, c.kv64, c.do64, c.o64, c.lse64, inp["topk"], c.scale, rows,
                              r_chunk=spec.r_chunk or None)
    compare(f"{name} dkv[sampled rows]", to_f64(dkv[torch.from_numpy(rows).cuda()]), ref_dkv)

    if c.sink is not None:
        compare(f"{name} d_sink", to_f64(dsink), c.ref_dsink())
    else:
        assert dsink is None


def test_full_size_forward(big):
    name, spec, inp, c = big
    o1, lse1 = smla.sparse_mla_fwd(c.q, c.kv, c.topk, c.sink, scale=c.scale)
    o2, lse2 = smla.sparse_mla_fwd(c.q, c.kv, c.topk, c.sink, scale=c.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2), "run-to-run results differ"
    # c.o64 is the oracle's O rounded to bf16, c.lse64 its lse rounded to fp32
    compare(f"{name} O", to_f64(o1), c.o64, cos_min=0.99999, rel=1e-2)
    assert np.max(np.abs(to_f64(lse1) - c.lse64)) < 1e-4
