"""CPU check of the derived zero-reference bound used by the GPU parity tests.

For topk = 1 without a sink the exact dq is zero, and the GPU's dq is fp32
rounding noise from forming dP and delta in different orders. This test
forms both sums in float32 in several orders (sequential, reversed, pairwise,
blocked like a warp reduction) and checks that the resulting dq stays inside
Case.dq_zero_bound, so the bound is not vacuous in the other direction either:
the noise must be nonzero somewhere.
"""

import numpy as np

from gpu_helpers import Case, custom_inputs


def _orders(x):
    """fp32 sums of the last axis of x in four different orders."""
    x = x.astype(np.float32)
    seq = np.zeros(x.shape[:-1], np.float32)
    for d in range(x.shape[-1]):
        seq = seq + x[..., d]
    rev = np.zeros(x.shape[:-1], np.float32)
    for d in range(x.shape[-1] - 1, -1, -1):
        rev = rev + x[..., d]
    pw = x
    while pw.shape[-1] > 1:
        pw = (pw[..., 0::2] + pw[..., 1::2]).astype(np.float32)
    blk = x.reshape(*x.shape[:-1], 32, 16)
    part = np.zeros(blk.shape[:-1], np.float32)
    for d in range(16):
        part = part + blk[..., d]
    while part.shape[-1] > 1:
        part = (part[..., 0::2] + part[..., 1::2]).astype(np.float32)
    return [seq, rev, pw[..., 0], part[..., 0]]


def test_dq_zero_bound_covers_fp32_reordering():
    c = Case(custom_inputs(11, T=12, H=16, K=1, N=20, sink=False, mask_p=0.0), device="cpu")
    bound = c.dq_zero_bound()
    idx = c.inp["topk"][:, 0]
    kvr = c.kv64[idx]
    prod = (c.do64 * kvr[:, None, :])            # exact in fp64 (bf16 x bf16)
    sums = _orders(prod)
    worst_noise = 0.0
    for a in sums:
        for b in sums:
            ds = np.float32(c.scale) * (a - b)                           # P = 1
            dq = ds.astype(np.float64)[:, :, None] * kvr[:, None, :]
            assert np.all(np.abs(dq) <= bound)
            worst_noise = max(worst_noise, float(np.max(np.abs(dq))))
    assert worst_noise > 0.0
    # the bound is a worst case: well above the typical noise, but not absurdly so
    assert np.max(bound) < 0.05
