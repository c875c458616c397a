"""Host-side checks of the seeded input recipe and of the FLOP convention."""

import json
import os

import numpy as np
import pytest

from sparse_mla_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_flop_convention_reproduces_printed_table():
    g = json.load(open(os.path.join(GOLDEN, "p1_performance_table.json")))
    w = g["workload"]
    flops = W.flops_nominal(w["T"], w["H"], w["topk"], w["D"])
    for row in g["rows"]:
        tflops = flops / (row["ms"] * 1e-3) / 1e12
        assert round(tflops) == row["tflops"], row


def test_tiny_window_layout():
    inp = W.make_inputs(W.WORKLOADS["tiny"])
    tk = inp["topk"]
    for t in (0, 5, 63, 64, 127):
        lo = max(0, t - 63)
        n = t - lo + 1
        assert np.array_equal(tk[t, :n], np.arange(lo, t + 1))
        assert np.all(tk[t, n:] == -1)
    assert W.valid_ranks(tk) == 6176


@pytest.mark.parametrize("name", ["t1024_h64"])
def test_window_plus_uniform_pool(name):
    s = W.WORKLOADS[name]
    inp = W.make_inputs(s)
    tk = inp["topk"]
    assert tk.shape == (s.T, s.topk) and tk.dtype == np.int32
    for t in (0, 10, 127, 128, 600, s.T - 1):
        row = tk[t]
        nwin = min(t + 1, s.window)
        assert np.array_equal(row[:nwin], np.arange(t - nwin + 1, t + 1))
        pool = row[nwin:nwin + s.pool_picks]
        assert np.all(np.diff(pool) > 0)
        assert pool.min() >= s.T and pool.max() < s.num_kv
        assert np.all(row[nwin + s.pool_picks:] == -1)
    assert inp["sink"].dtype == np.float32 and inp["sink"].shape == (s.H,)


def test_zipf_masked_workload_structure():
    s = W.WORKLOADS["t8192_zipf"]
    rng = np.random.Generator(np.random.PCG64(3))
    tk = W.make_topk(s, rng)
    frac = np.count_nonzero(tk < 0) / tk.size
    # 30 % random masking on top of the (few) short-window slots
    assert 0.29 < frac < 0.32
    pool_counts = np.bincount(tk[tk >= s.T] - s.T, minlength=s.pool_rows)
    # skew: the first pool rank is picked by nearly every token (before masking)
    assert pool_counts[0] > 0.6 * s.T
    assert pool_counts[0] > 3 * np.median(pool_counts)
    assert pool_counts[:50].min() > 5 * pool_counts[-50:].max()


def test_inputs_are_seeded_and_independent():
    s = W.WORKLOADS["tiny"]
    a = W.make_inputs(s, seed=0)
    b = W.make_inputs(s, seed=0)
    c = W.make_inputs(s, seed=1)
    for k in ("q", "kv", "do", "topk"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["q"], c["q"])
    # bf16 bit patterns of finite N(0,1) draws
    x = (a["q"].astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isfinite(x)) and 0.9 < x.std() < 1.1


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 3.0e-3], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even mantissa (1.0)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2**-6
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2**-8
