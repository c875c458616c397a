"""Pins of the fp64 oracle against things other than itself (CPU only).

The aiter page that defines the operation ("[WIP][TRITON][GLUON][GFX950]
[DSV4] Sparse MLA training backward") prints no worked numeric example, so
the oracle is pinned by:

* torch float64 autograd through an independently written dense-masked
  forward (gather + masked softmax with an extra sink logit column);
* central finite differences of L = sum(O * G) in float64;
* closed forms (topk = 1; all scores equal) and invariants (softmax mass
  with the sink is 1; masked and permuted ranks change nothing);
* the two dkv formulations (scatter vs inverted-CSR gather);
* brute force for the CSR.

Each check is chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""

import numpy as np
import pytest
import torch


def _rand_case(rng, T=5, H=3, D=8, K=6, N=9, sink=True, mask_p=0.25, dup=True):
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((N, D))
    do = rng.standard_normal((T, H, D))
    topk = rng.integers(0, N, size=(T, K)).astype(np.int32)
    if dup:
        topk[0, 1] = topk[0, 0]               # a duplicate slot
    topk[rng.random((T, K)) < mask_p] = -1
    topk[1, 0] = 2                             # keep at least one valid rank here
    s = rng.standard_normal(H) if sink else None
    return q, kv, do, topk, s


def _torch_reference(q, kv, do, topk, sink, scale):
    """Dense-masked forward written with torch ops; autograd gives the grads."""
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kvt = torch.tensor(kv, dtype=torch.float64, requires_grad=True)
    idx = torch.tensor(topk, dtype=torch.int64)
    valid = idx >= 0
    g = kvt[idx.clamp(min=0)]                                   # [T, K, D]
    s = torch.einsum("thd,tkd->thk", qt, g) * scale
    s = s.masked_fill(~valid[:, None, :], float("-inf"))
    st = None
    if sink is not None:
        st = torch.tensor(sink, dtype=torch.float64, requires_grad=True)
        col = st[None, :, None].expand(s.shape[0], s.shape[1], 1)
        logits = torch.cat([s, col], dim=-1)
    else:
        logits = s
    lse = torch.logsumexp(logits, dim=-1)
    p = torch.exp(logits - lse[..., None])[..., : s.shape[-1]]
    o = torch.einsum("thk,tkd->thd", p, g)
    loss = (o * torch.tensor(do)).sum()
    loss.backward()
    return {
        "o": o.detach().numpy(), "lse": lse.detach().numpy(),
        "dq": qt.grad.numpy(), "dkv": kvt.grad.numpy(),
        "dsink": None if st is None else st.grad.numpy(),
    }


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("with_sink", [True, False])
def test_dense_case_matches_torch_autograd(oracle_mod, with_sink):
    """topk = all rows (permuted per token): textbook MQA attention (+ sink column)."""
    rng = np.random.default_rng(1)
    T, H, D = 6, 3, 8
    N = T
    q = rng.standard_normal((T, H, D)); kv = rng.standard_normal((N, D))
    do = rng.standard_normal((T, H, D))
    topk = np.stack([rng.permutation(N) for _ in range(T)]).astype(np.int32)
    sink = rng.standard_normal(H) if with_sink else None
    scale = 1 / np.sqrt(D)
    ref = _torch_reference(q, kv, do, topk, sink, scale)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    assert _rel(o, ref["o"]) < 1e-12 and _rel(lse, ref["lse"]) < 1e-12
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    assert _rel(g["dq"], ref["dq"]) < 1e-11
    assert _rel(g["dkv"], ref["dkv"]) < 1e-11
    if with_sink:
        assert _rel(g["dsink"], ref["dsink"]) < 1e-11
    else:
        assert g["dsink"] is None


@pytest.mark.parametrize("with_sink", [True, False])
def test_sparse_masked_duplicates_match_torch_autograd(oracle_mod, with_sink):
    """-1 slots, duplicate indices, pool rows never referenced, D=512."""
    rng = np.random.default_rng(2)
    q, kv, do, topk, sink = _rand_case(rng, T=7, H=4, D=512, K=10, N=13,
                                       sink=with_sink)
    scale = 1 / np.sqrt(512)
    ref = _torch_reference(q, kv, do, topk, sink, scale)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    assert _rel(o, ref["o"]) < 1e-12 and _rel(lse, ref["lse"]) < 1e-12
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    for k in ("dq", "dkv") + (("dsink",) if with_sink else ()):
        assert _rel(g[k], ref[k]) < 1e-11, k


def test_finite_differences(oracle_mod):
    """Central differences of L = sum(O*G) against the backward (exact O, lse)."""
    rng = np.random.default_rng(3)
    q, kv, do, topk, sink = _rand_case(rng, T=4, H=2, D=6, K=5, N=7)
    scale = 0.37

    def loss(q_, kv_, s_):
        o, _ = oracle_mod.fwd(q_, kv_, topk, s_, scale)
        return float(np.sum(o * do))

    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    eps = 1e-6

    def fd(arr, fn):
        out = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            a1 = arr.copy(); a1[i] += eps
            a0 = arr.copy(); a0[i] -= eps
            out[i] = (fn(a1) - fn(a0)) / (2 * eps)
        return out

    fq = fd(q, lambda a: loss(a, kv, sink))
    fkv = fd(kv, lambda a: loss(q, a, sink))
    fs = fd(sink, lambda a: loss(q, kv, a))
    assert _rel(g["dq"], fq) < 1e-7
    assert _rel(g["dkv"], fkv) < 1e-7
    assert _rel(g["dsink"], fs) < 1e-7
    # kv rows that no valid slot references get exactly zero gradient
    used = set(int(j) for j in topk.ravel() if j >= 0)
    for j in range(kv.shape[0]):
        if j not in used:
            assert np.all(g["dkv"][j] == 0.0)


def test_dsink_identity(oracle_mod):
    """d_sink_h = -sum_t exp(sink_h - lse) * delta, computed two ways."""
    rng = np.random.default_rng(4)
    q, kv, do, topk, sink = _rand_case(rng, T=6, H=3, D=16, K=6, N=8)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, 0.25)
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, 0.25)
    ds, delta = oracle_mod.dsink(do, o, lse, sink)
    assert np.allclose(delta, np.einsum("thd,thd->th", o, do), rtol=1e-13, atol=1e-13)
    assert _rel(g["dsink"], ds) < 1e-13


def test_softmax_mass_with_sink_is_one(oracle_mod):
    """With q = kv rows one-hot, O picks out the softmax weights directly."""
    rng = np.random.default_rng(5)
    T, H, K = 3, 2, 5
    N = D = 8
    kv = np.eye(N)                       # kv row j = e_j, so O[d] = sum of P over slots of row d
    q = rng.standard_normal((T, H, D))
    topk = np.stack([rng.permutation(N)[:K] for _ in range(T)]).astype(np.int32)
    topk[2, 3] = -1
    sink = rng.standard_normal(H)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, 0.7)
    mass = o.sum(-1) + np.exp(sink[None, :] - lse)
    assert np.allclose(mass, 1.0, rtol=0, atol=1e-14)


def test_uniform_scores_closed_form(oracle_mod):
    """q = 0: every valid score is 0, lse = log(n + e^sink), O = mean * n/(n+e^sink)."""
    rng = np.random.default_rng(6)
    T, H, D, K, N = 4, 2, 8, 6, 10
    q = np.zeros((T, H, D)); kv = rng.standard_normal((N, D))
    topk = rng.integers(0, N, size=(T, K)).astype(np.int32)
    topk[:, -2:] = -1
    sink = np.array([0.3, -1.2])
    o, lse = oracle_mod.fwd(q, kv, topk, sink, 1 / np.sqrt(512))
    for t in range(T):
        rows = topk[t][topk[t] >= 0]
        n = rows.size
        for h in range(H):
            assert abs(lse[t, h] - np.log(n + np.exp(sink[h]))) < 1e-14
            expect = kv[rows].sum(0) / (n + np.exp(sink[h]))
            assert np.max(np.abs(o[t, h] - expect)) < 1e-14


def test_topk1_closed_forms(oracle_mod):
    """topk = 1: without a sink O = kv[idx], dq = 0, dkv[idx] = sum dO; with a sink P = sigmoid."""
    rng = np.random.default_rng(7)
    T, H, D, N = 5, 3, 8, 6
    q = rng.standard_normal((T, H, D)); kv = rng.standard_normal((N, D))
    do = rng.standard_normal((T, H, D))
    topk = rng.integers(0, N, size=(T, 1)).astype(np.int32)
    scale = 0.5
    o, lse = oracle_mod.fwd(q, kv, topk, None, scale)
    assert np.array_equal(o, np.broadcast_to(kv[topk[:, 0]][:, None, :], o.shape))
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, None, scale)
    assert np.max(np.abs(g["dq"])) < 1e-13
    expect = np.zeros((N, D))
    for t in range(T):
        expect[topk[t, 0]] += do[t].sum(0)
    assert np.max(np.abs(g["dkv"] - expect)) < 1e-12

    sink = rng.standard_normal(H)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    for t in range(T):
        j = topk[t, 0]
        for h in range(H):
            s = scale * q[t, h] @ kv[j]
            p = 1.0 / (1.0 + np.exp(sink[h] - s))
            assert np.allclose(o[t, h], p * kv[j], rtol=1e-13, atol=1e-14)
            dp = do[t, h] @ kv[j]
            # dS = P (dP - delta) with delta = O.dO = P dP  =>  dS = P(1-P) dP
            expect_dq = scale * p * (1 - p) * dp * kv[j]
            assert np.allclose(g["dq"][t, h], expect_dq, rtol=1e-11, atol=1e-13)


def test_mask_and_permutation_invariance(oracle_mod):
    """Adding -1 slots or permuting ranks leaves every output unchanged."""
    rng = np.random.default_rng(8)
    q, kv, do, topk, sink = _rand_case(rng, T=5, H=2, D=16, K=6, N=9)
    scale = 0.3
    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    perm = np.stack([rng.permutation(topk.shape[1]) for _ in range(topk.shape[0])])
    tk2 = np.take_along_axis(topk, perm, axis=1)
    tk2 = np.concatenate([tk2, -np.ones((tk2.shape[0], 3), np.int32)], axis=1)
    tk2 = np.ascontiguousarray(np.roll(tk2, 2, axis=1))
    o2, lse2 = oracle_mod.fwd(q, kv, tk2, sink, scale)
    assert _rel(o2, o) < 1e-13 and _rel(lse2, lse) < 1e-13
    g2 = oracle_mod.bwd(q, kv, do, o, lse, tk2, sink, scale)
    for k in ("dq", "dkv", "dsink"):
        assert _rel(g2[k], g[k]) < 1e-12, k


def test_row_without_valid_rank(oracle_mod):
    """All slots masked: O = 0, lse = sink (or -inf), no NaN, zero gradient."""
    rng = np.random.default_rng(9)
    q, kv, do, topk, sink = _rand_case(rng, T=4, H=2, D=8, K=4, N=6, mask_p=0.0)
    topk[2, :] = -1
    for s in (sink, None):
        o, lse = oracle_mod.fwd(q, kv, topk, s, 0.5)
        assert np.all(o[2] == 0.0)
        if s is None:
            assert np.all(np.isneginf(lse[2]))
        else:
            assert np.array_equal(lse[2], s)
        g = oracle_mod.bwd(q, kv, do, o, lse, topk, s, 0.5)
        assert np.all(g["dq"][2] == 0.0)
        assert np.all(np.isfinite(g["dq"])) and np.all(np.isfinite(g["dkv"]))
        if s is not None:
            # the masked token adds exp(sink - sink) * delta with delta = O.dO = 0
            other = oracle_mod.bwd(q[[0, 1, 3]], kv, do[[0, 1, 3]], o[[0, 1, 3]],
                                   lse[[0, 1, 3]], topk[[0, 1, 3]], s, 0.5)
            assert _rel(g["dsink"], other["dsink"]) < 1e-14


def test_scatter_equals_csr_gather(oracle_mod):
    """dkv by scatter over (t, r) equals dkv gathered per kv row through the CSR."""
    rng = np.random.default_rng(10)
    q, kv, do, topk, sink = _rand_case(rng, T=9, H=3, D=32, K=8, N=12)
    scale = 1 / np.sqrt(32)
    o, lse = oracle_mod.fwd(q, kv, topk, sink, scale)
    g = oracle_mod.bwd(q, kv, do, o, lse, topk, sink, scale)
    rows = np.arange(kv.shape[0])
    for r_chunk in (None, 4, 2):
        dk = oracle_mod.dkv_rows(q, kv, do, o, lse, topk, scale, rows, r_chunk=r_chunk)
        assert _rel(dk, g["dkv"]) < 1e-12
    dq = oracle_mod.dq_tokens(q, kv, do, o, lse, topk, scale, [0, 4, 8])
    assert _rel(dq, g["dq"][[0, 4, 8]]) < 1e-13


def _csr_brute(topk, N, r0, R):
    pairs = []
    T = topk.shape[0]
    for t in range(T):
        for r in range(r0, r0 + R):
            j = int(topk[t, r])
            if j >= 0:
                pairs.append((j, t * R + (r - r0)))
    pairs.sort()
    row_ptr = np.zeros(N + 1, dtype=np.int64)
    for j, _ in pairs:
        row_ptr[j + 1] += 1
    return np.cumsum(row_ptr), np.array([p for _, p in pairs], dtype=np.int64)


@pytest.mark.parametrize("r0,R", [(0, 7), (0, 3), (3, 4), (6, 1)])
def test_csr_brute_force(oracle_mod, r0, R):
    rng = np.random.default_rng(11)
    T, K, N = 11, 7, 9
    topk = rng.integers(-1, N, size=(T, K)).astype(np.int32)
    topk[0, :3] = 4                                  # duplicates in one row
    rp, col = oracle_mod.csr(topk, N, r0, R)
    brp, bcol = _csr_brute(topk, N, r0, R)
    assert np.array_equal(rp, brp) and np.array_equal(col, bcol)
    # invariants
    assert np.all(np.diff(rp) >= 0)
    assert rp[-1] == np.count_nonzero(topk[:, r0:r0 + R] >= 0)
    for j in range(N):
        seg = col[rp[j]:rp[j + 1]]
        assert np.all(np.diff(seg) > 0)
        for p in seg:
            assert topk[p // R, r0 + p % R] == j


def test_out_of_range_index_is_an_error(oracle_mod):
    rng = np.random.default_rng(12)
    q, kv, do, topk, sink = _rand_case(rng)
    bad = topk.copy(); bad[1, 1] = kv.shape[0]
    with pytest.raises(RuntimeError):
        oracle_mod.fwd(q, kv, bad, sink, 0.5)
    bad[1, 1] = -2
    with pytest.raises(RuntimeError):
        oracle_mod.csr(bad, kv.shape[0])
