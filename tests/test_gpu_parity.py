"""GPU parity of the CUDA path against the fp64 oracle (small and medium sizes,
full tensors), plus edge cases, determinism and chunking.

Every call goes through the C ABI (sparse_mla_attention_gb300.api marshals
torch tensors into libsmla.so).
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_gb300 as smla
from sparse_mla_attention_gb300 import _lib, workloads as W
from gpu_helpers import Case, compare, custom_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mla_attention_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def tiny():
    return Case(W.make_inputs(W.WORKLOADS["tiny"]))


@pytest.fixture(scope="module")
def t1024():
    return Case(W.make_inputs(W.WORKLOADS["t1024_h64"]))


def _run_bwd(c: Case, r_chunk=None, ws=None, out=None):
    return smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, scale=c.scale,
                               r_chunk=r_chunk, workspace=ws, out=out)


def _check_full(c: Case, r_chunk=None):
    dq, dkv, dsink = _run_bwd(c, r_chunk)
    ref = c.ref_full()
    zb = c.dq_zero_bound() if not np.any(ref["dq"]) and c.K == 1 and c.sink is None else None
    compare("dq", to_f64(dq), ref["dq"], zero_bound=zb)
    compare("dkv", to_f64(dkv), ref["dkv"])
    if c.sink is not None:
        compare("d_sink", to_f64(dsink), ref["dsink"])
    else:
        assert dsink is None


# ------------------------------------------------------------------- CSR
@pytest.mark.parametrize("name,r0,r_len", [
    ("tiny", 0, 64), ("tiny", 16, 16), ("t1024_h64", 0, 256), ("t1024_h64", 128, 128),
    ("headline", 0, 512), ("headline", 384, 128), ("t8192_zipf", 0, 512),
])
def test_csr_bit_exact(name, r0, r_len):
    spec = W.WORKLOADS[name]
    rng = np.random.Generator(np.random.PCG64(5))
    topk = W.make_topk(spec, rng)
    rp, col = smla.csr_build(torch.from_numpy(topk).cuda(), spec.num_kv, r0, r_len)
    erp, ecol = oracle.csr(topk, spec.num_kv, r0, r_len)
    assert np.array_equal(rp.cpu().numpy(), erp)
    assert np.array_equal(col.cpu().numpy(), ecol)


def test_csr_edge_cases():
    rng = np.random.default_rng(0)
    topk = rng.integers(-1, 7, size=(33, 9)).astype(np.int32)
    topk[0, :] = 3                          # one row referenced 9 times by one token
    topk[5, :] = -1
    for r0, R in ((0, 9), (2, 3), (8, 1)):
        rp, col = smla.csr_build(torch.from_numpy(topk).cuda(), 7, r0, R)
        erp, ecol = oracle.csr(topk, 7, r0, R)
        assert np.array_equal(rp.cpu().numpy(), erp) and np.array_equal(col.cpu().numpy(), ecol)
    # no valid entry at all, and no token at all
    rp, col = smla.csr_build(torch.full((4, 5), -1, dtype=torch.int32, device="cuda"), 6)
    assert rp.cpu().tolist() == [0] * 7 and col.numel() == 0
    rp, col = smla.csr_build(torch.zeros((0, 5), dtype=torch.int32, device="cuda"), 6)
    assert rp.cpu().tolist() == [0] * 7


# --------------------------------------------------------------- forward
def test_forward_matches_oracle(tiny):
    o, lse = smla.sparse_mla_fwd(tiny.q, tiny.kv, tiny.topk, tiny.sink, scale=tiny.scale)
    _, _, o64, lse64 = oracle.fwd_inputs(tiny.inp)
    compare("o", to_f64(o), o64, cos_min=0.99999, rel=1e-2)
    assert np.max(np.abs(to_f64(lse) - lse64)) < 1e-4


def test_forward_no_sink_and_masked_rows():
    c = custom_inputs(1, T=9, H=16, K=40, N=50, sink=False, all_masked_rows=(3,))
    case = Case(c)
    o, lse = smla.sparse_mla_fwd(case.q, case.kv, case.topk, None, scale=case.scale)
    o64, lse64 = oracle.fwd(case.q64, case.kv64, c["topk"], None, case.scale)
    lse_g = to_f64(lse)
    assert np.all(np.isneginf(lse_g[3])) and np.all(to_f64(o)[3] == 0)
    ok = np.isfinite(lse64)
    assert np.max(np.abs(lse_g[ok] - lse64[ok])) < 1e-4
    compare("o", to_f64(o), o64, cos_min=0.99999, rel=1e-2)


# (H, K, N, T, sink): H a multiple of 32 with topk <= 512 runs on the tensor
# cores, the other shapes on the CUDA-core kernel
@pytest.mark.parametrize("H,K,N,T,sink", [
    (32, 48, 90, 70, True),         # one ragged rank tile
    (64, 200, 260, 130, False),     # two tiles, no sink
    (96, 1, 20, 12, True),          # topk = 1
    (128, 512, 700, 40, True),      # four full rank tiles
    (128, 300, 520, 400, False),    # more tokens than SMs: the persistent loop
    (64, 129, 300, 160, True),      # one rank past a tile boundary
    (48, 80, 100, 30, True),        # H not a multiple of 32: CUDA-core kernel
    (32, 600, 700, 20, True),       # topk > 512: CUDA-core kernel
])
def test_forward_shapes(H, K, N, T, sink):
    c = custom_inputs(H * 11 + K, T=T, H=H, K=K, N=N, sink=sink,
                      all_masked_rows=(min(2, T - 1),))
    case = Case(c)
    o_out = torch.full_like(case.q, float("nan"))
    lse_out = torch.full((T, H), float("nan"), device="cuda")
    o, lse = smla.sparse_mla_fwd(case.q, case.kv, case.topk, case.sink, scale=case.scale,
                                 out=(o_out, lse_out))
    o64, lse64 = oracle.fwd(case.q64, case.kv64, c["topk"], case.sink64, case.scale)
    o_g, lse_g = to_f64(o), to_f64(lse)
    m = min(2, T - 1)                       # the fully masked token
    assert np.all(o_g[m] == 0)
    if sink:
        assert np.array_equal(lse_g[m], case.sink64)    # lse = sink exactly
    else:
        assert np.all(np.isneginf(lse_g[m]))
    ok = np.isfinite(lse64)
    assert np.array_equal(ok, np.isfinite(lse_g))
    assert np.max(np.abs(lse_g[ok] - lse64[ok])) < 1e-4
    compare("o", o_g, o64, cos_min=0.99999, rel=1e-2)


@pytest.mark.parametrize("H", [16, 32, 128])
def test_forward_topk1_no_sink_is_exact(H):
    # One valid rank and no sink: the softmax weight is exactly 1, so O is the
    # selected kv row bit for bit and lse is that rank's score (both kernels:
    # H = 16 runs on CUDA cores, H = 32 and 128 on the tensor cores).
    T, N = 200, 300
    c = custom_inputs(H, T=T, H=H, K=1, N=N, sink=False, mask_p=0.0)
    case = Case(c)
    o, lse = smla.sparse_mla_fwd(case.q, case.kv, case.topk, None, scale=case.scale)
    idx = torch.from_numpy(c["topk"][:, 0].astype(np.int64)).cuda()
    want = case.kv[idx].unsqueeze(1).expand(T, H, 512)
    assert torch.equal(o, want)
    s64 = np.einsum("thd,td->th", case.q64, case.kv64[c["topk"][:, 0]]) * case.scale
    assert np.max(np.abs(to_f64(lse) - s64)) < 1e-4


def test_forward_after_backward_h32():
    # The tensor-core forward runs M = 128 MMAs whatever H is; the TMEM lanes of
    # heads >= H then hold scores of stale shared memory (the previous kernel's
    # bytes). They must not change control flow: run the backward first so that
    # shared memory holds its data, then the forward.
    c = custom_inputs(91, T=300, H=32, K=256, N=400, sink=True, all_masked_rows=(7,))
    case = Case(c)
    for _ in range(2):
        smla.sparse_mla_bwd(case.q, case.kv, case.do, case.o, case.lse, case.topk, case.sink,
                            scale=case.scale)
        o, lse = smla.sparse_mla_fwd(case.q, case.kv, case.topk, case.sink, scale=case.scale)
        compare("o", to_f64(o), case.o64, cos_min=0.99999, rel=1e-2)
        assert np.max(np.abs(to_f64(lse) - case.lse64)) < 1e-4


def test_forward_t1024(t1024):
    o1, lse1 = smla.sparse_mla_fwd(t1024.q, t1024.kv, t1024.topk, t1024.sink, scale=t1024.scale)
    o2, lse2 = smla.sparse_mla_fwd(t1024.q, t1024.kv, t1024.topk, t1024.sink, scale=t1024.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    # t1024.o64 / lse64: the oracle's forward rounded to bf16 / fp32
    compare("o", to_f64(o1), t1024.o64, cos_min=0.99999, rel=1e-2)
    assert np.max(np.abs(to_f64(lse1) - t1024.lse64)) < 1e-4


@pytest.mark.parametrize("H", [16, 32])
def test_forward_out_of_range_index_reports_and_masks(H):
    c = custom_inputs(4, T=8, H=H, K=12, N=20, sink=True, mask_p=0.0)
    case = Case(c)
    bad = case.topk.clone()
    bad[4, 5] = 20          # == num_kv: out of range
    bad[6, 0] = -7
    with pytest.raises(_lib.SmlaError) as e:
        smla.sparse_mla_fwd(case.q, case.kv, bad, case.sink, scale=case.scale)
    assert e.value.code == _lib.SMLA_ERR_INDEX
    masked = bad.clone(); masked[4, 5] = -1; masked[6, 0] = -1
    r1 = smla.sparse_mla_fwd(case.q, case.kv, bad, case.sink, scale=case.scale, check_status=False)
    r2 = smla.sparse_mla_fwd(case.q, case.kv, masked, case.sink, scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])


def test_forward_empty_T():
    q = torch.zeros((0, 64, 512), dtype=torch.bfloat16, device="cuda")
    kv = torch.randn((10, 512), device="cuda").bfloat16()
    topk = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    o, lse = smla.sparse_mla_fwd(q, kv, topk, None)
    assert o.numel() == 0 and lse.numel() == 0


# -------------------------------------------------------------- backward
def test_bwd_tiny_full(tiny):
    _check_full(tiny)


def test_bwd_t1024_full(t1024):
    _check_full(t1024)


def test_bwd_t1024_chunked_matches_unchunked(t1024):
    dq1, dkv1, ds1 = _run_bwd(t1024)
    dq2, dkv2, ds2 = _run_bwd(t1024, r_chunk=64)
    compare("dq chunked", to_f64(dq2), to_f64(dq1), cos_min=0.99999, rel=1e-2)
    compare("dkv chunked", to_f64(dkv2), to_f64(dkv1), cos_min=0.99999, rel=1e-2)
    assert torch.equal(ds1, ds2)
    ref = t1024.ref_full()
    compare("dq", to_f64(dq2), ref["dq"])
    compare("dkv", to_f64(dkv2), ref["dkv"])


@pytest.mark.parametrize("H,K,N,T,sink,chunk", [
    (16, 1, 20, 12, True, 0),       # topk = 1
    (16, 1, 20, 12, False, 0),
    (32, 48, 90, 70, True, 16),     # ragged tiles, chunks
    (64, 200, 260, 130, False, 40), # several rank tiles, no sink, uneven chunk
    (128, 72, 150, 37, True, 0),
    (48, 100, 150, 40, True, 0),    # the head counts between: odd 16-head chunks,
    (80, 64, 90, 33, False, 32),    # 64-head stash padding (48), 128-head padding
    (96, 256, 300, 160, True, 128), # (80, 96, 112), more tokens than SMs (160)
    (112, 130, 200, 21, True, 0),
    (48, 100, 150, 41, True, 0),    # two-token items (heads <= 64, <= 128 ranks), odd T:
    (16, 256, 300, 33, False, 64),  # the last item has one token; unchunked and chunked
])
def test_bwd_custom_shapes(H, K, N, T, sink, chunk):
    c = Case(custom_inputs(H * 7 + K, T=T, H=H, K=K, N=N, sink=sink,
                           all_masked_rows=(min(2, T - 1),), r_chunk=chunk))
    _check_full(c, r_chunk=chunk or None)


@pytest.mark.parametrize("H,K,N,T,sink,chunk,mask_p", [
    (128, 512, 700, 45, True, 0, 0.1),     # two 256-rank items per token, masked slots compacted
    (128, 600, 900, 23, True, 0, 0.0),     # a third, ragged item (88 ranks)
    (64, 384, 500, 50, False, 0, 0.3),     # the second item has one tile
    (96, 520, 640, 31, True, 0, 0.05),     # 8 ranks in the third item
    (128, 640, 800, 17, True, 320, 0.1),   # two rank chunks of 320 (per-chunk dq)
    (112, 257, 300, 40, False, 0, 0.0),    # one rank past two tiles
])
def test_bwd_many_rank_items(H, K, N, T, sink, chunk, mask_p):
    """Tokens with more than 256 ranks (per chunk) span several S/dP/dS items:
    ragged last items, items of one tile or a few ranks, masked slots that
    compaction moves to the end, and rank chunks wider than 256."""
    c = Case(custom_inputs(H * 5 + K, T=T, H=H, K=K, N=N, sink=sink, mask_p=mask_p,
                           all_masked_rows=(min(3, T - 1),), r_chunk=chunk))
    _check_full(c, r_chunk=chunk or None)


@pytest.mark.parametrize("H,K,N,T", [(64, 200, 260, 130), (128, 300, 400, 20)])
def test_bwd_q_do_placement(H, K, N, T):
    """q and dO are fetched as one paired tensor when one sits below the other
    in memory (either order), and as two separate tensors when they coincide.
    All three give the oracle's gradients; the two paired orders run the same
    arithmetic on permuted accumulator columns, so their results are equal bit
    for bit."""
    c = Case(custom_inputs(H * 3 + K, T=T, H=H, K=K, N=N, sink=True, all_masked_rows=(1,)))
    ref = c.ref_full()
    outs = []
    for q_first in (True, False):
        buf = torch.empty((2,) + tuple(c.q.shape), dtype=torch.bfloat16, device="cuda")
        q, do = (buf[0], buf[1]) if q_first else (buf[1], buf[0])
        q.copy_(c.q)
        do.copy_(c.do)
        assert (q.data_ptr() < do.data_ptr()) == q_first
        outs.append(smla.sparse_mla_bwd(q, c.kv, do, c.o, c.lse, c.topk, c.sink, scale=c.scale))
        compare("dq", to_f64(outs[-1][0]), ref["dq"])
        compare("dkv", to_f64(outs[-1][1]), ref["dkv"])
        compare("d_sink", to_f64(outs[-1][2]), ref["dsink"])
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    # dO is q itself (one tensor passed twice): separate loads
    dq, dkv, ds = smla.sparse_mla_bwd(c.q, c.kv, c.q, c.o, c.lse, c.topk, c.sink, scale=c.scale)
    ref2 = oracle.bwd(c.q64, c.kv64, c.q64, c.o64, c.lse64, c.inp["topk"], c.sink64, c.scale)
    compare("dq (dO = q)", to_f64(dq), ref2["dq"])
    compare("dkv (dO = q)", to_f64(dkv), ref2["dkv"])
    compare("d_sink (dO = q)", to_f64(ds), ref2["dsink"])


def test_bwd_valid_counts_on_tile_boundaries():
    """Each token's valid ranks are compacted before tiling: counts of 0, 1 and
    around every 64-rank chunk and 128-rank tile boundary, masked slots at
    random positions, duplicate indices kept."""
    counts = [0, 1, 2, 63, 64, 65, 127, 128, 129, 191, 192, 255, 256, 257, 300, 383, 384, 385, 400]
    T, H, K, N = len(counts), 64, 400, 700
    c = custom_inputs(991, T=T, H=H, K=K, N=N, sink=True, mask_p=0.0)
    rng = np.random.default_rng(991)
    topk = c["topk"]
    for t, m in enumerate(counts):
        keep = np.zeros(K, dtype=bool)
        keep[rng.choice(K, size=m, replace=False)] = True
        topk[t, ~keep] = -1
    topk[3, np.flatnonzero(topk[3] >= 0)[:2]] = 5      # a duplicated row inside a token
    case = Case(c)
    _check_full(case)


def test_bwd_empty_T():
    H, N = 16, 10
    q = torch.zeros((0, H, 512), dtype=torch.bfloat16, device="cuda")
    kv = torch.randn((N, 512), device="cuda").bfloat16()
    topk = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    lse = torch.zeros((0, H), dtype=torch.float32, device="cuda")
    sink = torch.randn(H, device="cuda")
    dkv0 = torch.full_like(kv, float("nan"))
    dq, dkv, ds = smla.sparse_mla_bwd(q, kv, q, q, lse, topk, sink,
                                      out=(torch.empty_like(q), dkv0, torch.full((H,), 7.0, device="cuda")))
    assert dq.numel() == 0 and torch.all(dkv == 0) and torch.all(ds == 0)


def test_bwd_out_of_range_index_reports_and_masks():
    c = custom_inputs(3, T=8, H=16, K=12, N=20, sink=True, mask_p=0.0)
    case = Case(c)
    bad = case.topk.clone()
    bad[4, 5] = 20          # == num_kv: out of range
    bad[6, 0] = -7
    with pytest.raises(_lib.SmlaError) as e:
        smla.sparse_mla_bwd(case.q, case.kv, case.do, case.o, case.lse, bad, case.sink)
    assert e.value.code == _lib.SMLA_ERR_INDEX
    # results equal those with the bad slots masked
    masked = bad.clone(); masked[4, 5] = -1; masked[6, 0] = -1
    r1 = smla.sparse_mla_bwd(case.q, case.kv, case.do, case.o, case.lse, bad, case.sink,
                             check_status=False)
    r2 = smla.sparse_mla_bwd(case.q, case.kv, case.do, case.o, case.lse, masked, case.sink)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_bwd_nan_poisoned_outputs_and_workspace(t1024):
    """Every output cell must be written; stale workspace bytes must not leak in."""
    ws = smla.Workspace()
    dims = smla.make_dims(t1024.T, t1024.H, t1024.K, t1024.N)
    buf = ws.get(smla.workspace_size(_lib.SMLA_OP_BWD, dims))
    buf.fill_(0xFF)
    dq = torch.full_like(t1024.q, float("nan"))
    dkv = torch.full_like(t1024.kv, float("nan"))
    ds = torch.full((t1024.H,), float("nan"), device="cuda")
    _run_bwd(t1024, ws=ws, out=(dq, dkv, ds))
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dkv.float()).all()
    assert torch.isfinite(ds).all()
    dq2, dkv2, ds2 = _run_bwd(t1024)
    assert torch.equal(dq, dq2) and torch.equal(dkv, dkv2) and torch.equal(ds, ds2)


def test_bwd_bitwise_deterministic(t1024):
    ws = smla.Workspace()
    runs = [_run_bwd(t1024, ws=ws) for _ in range(3)] + [_run_bwd(t1024)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    runs = [_run_bwd(t1024, r_chunk=128, ws=ws) for _ in range(2)]
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)


def test_bwd_rejects_bad_input_on_host(t1024):
    with pytest.raises(TypeError):
        smla.sparse_mla_bwd(t1024.q.float(), t1024.kv, t1024.do, t1024.o, t1024.lse, t1024.topk)
    with pytest.raises(ValueError):
        smla.sparse_mla_bwd(t1024.q, t1024.kv, t1024.do, t1024.o, t1024.lse[:, :3], t1024.topk)
    with pytest.raises(_lib.SmlaError) as e:
        smla.sparse_mla_bwd(t1024.q, t1024.kv, t1024.do, t1024.o, t1024.lse, t1024.topk,
                            t1024.sink, r_chunk=100)
    assert e.value.code == _lib.SMLA_ERR_RCHUNK


def test_bwd_rejects_host_or_misshapen_out_tensors(t1024):
    c = t1024
    H = c.H
    good = (torch.empty_like(c.q), torch.empty_like(c.kv), torch.empty(H, device="cuda"))
    bad_outs = [
        (good[0].cpu(), good[1], good[2]),                       # dq on the host
        (good[0], good[1].cpu(), good[2]),                       # dkv on the host
        (good[0], good[1], good[2].cpu()),                       # d_sink on the host
        (good[0][:-1], good[1], good[2]),                        # dq one token short
        (good[0], good[1][:-1], good[2]),                        # dkv one row short
        (good[0], good[1], None),                                # d_sink missing with a sink
        (good[0].float(), good[1], good[2]),                     # wrong dtype
    ]
    for out in bad_outs:
        with pytest.raises((ValueError, TypeError)):
            smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, out=out)
    # nothing was launched: a following call is still correct
    dq, dkv, ds = smla.sparse_mla_bwd(c.q, c.kv, c.do, c.o, c.lse, c.topk, c.sink, out=good)
    compare("d_sink after refused calls", to_f64(ds), c.ref_dsink())


def test_c_abi_refuses_host_pointers(t1024):
    """A host pointer where device memory is required returns SMLA_ERR_DEVICE
    before anything is enqueued (it would fault the GPU inside a kernel)."""
    import ctypes
    c = t1024
    lib = _lib.load()
    T, H = c.T, c.H
    dims = smla.api.make_dims(T, H, c.K, c.N, 0, None)
    n = ctypes.c_size_t()
    assert lib.smla_workspace_size(_lib.SMLA_OP_BWD, ctypes.byref(dims), ctypes.byref(n)) == 0
    ws = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    dq, dkv = torch.empty_like(c.q), torch.empty_like(c.kv)
    ds = torch.empty(H, device="cuda")
    host_dq = torch.empty(c.q.shape, dtype=c.q.dtype, pin_memory=True)
    host_kv = torch.empty(c.kv.shape, dtype=c.kv.dtype)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def bwd(q=c.q, kv=c.kv, dq_=dq, dkv_=dkv):
        return lib.smla_bwd(p(q), p(kv), p(c.do), p(c.o), p(c.lse), p(c.topk), p(c.sink),
                            p(dq_), p(dkv_), p(ds), ctypes.byref(dims), p(ws), n.value, s)
    assert bwd(dq_=host_dq) == _lib.SMLA_ERR_DEVICE          # pinned host output
    assert bwd(kv=host_kv) == _lib.SMLA_ERR_DEVICE           # pageable host input
    assert lib.smla_dsink_static(p(c.do), p(c.o), p(c.lse), p(c.sink), p(host_dq), T, H, s) \
        == _lib.SMLA_ERR_DEVICE
    fdims = smla.api.make_dims(T, H, c.K, c.N, 0, None)
    o = torch.empty_like(c.q)
    host_lse = torch.empty((T, H), dtype=torch.float32)
    assert lib.smla_fwd(p(c.q), p(c.kv), p(c.topk), p(c.sink), p(o), p(host_lse),
                        ctypes.byref(fdims), p(ws), n.value, s) == _lib.SMLA_ERR_DEVICE
    torch.cuda.synchronize()
    assert bwd() == _lib.SMLA_OK
    torch.cuda.synchronize()
    compare("d_sink after refused calls", to_f64(ds), c.ref_dsink())
