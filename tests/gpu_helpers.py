"""Shared helpers of the GPU parity tests: device copies of the seeded inputs,
oracle references and the comparison bar.

The bar (for every floating-point output): cosine similarity > 0.999 and
max |gpu - ref| <= 2e-2 * max |ref|. Where the reference is identically zero
(dq when topk = 1 without a sink) the caller passes an elementwise bound
derived from fp32 rounding (Case.dq_zero_bound); without one, zeros must be
exact. The CSR is compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mla_attention_gb300 import workloads as W

COS_MIN = 0.999
MAXABS_REL = 2e-2
# Unit roundoff allowed for one fp32 addition on the GPU: 2^-23, twice IEEE
# round-to-nearest's 2^-24, so that adders that truncate (as tensor-core
# accumulation may) are covered as well.
FP32_U = 2.0 ** -23


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f64(bf16_bits(t))
    return t.detach().cpu().double().numpy()


def compare(name: str, got: np.ndarray, ref: np.ndarray, cos_min=COS_MIN, rel=MAXABS_REL,
            zero_bound=None):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    if scale == 0.0:
        # The reference is exactly zero. With a derived bound (zero_bound, same
        # shape as ref) every element must lie within it; without one, exactly 0.
        if zero_bound is None:
            assert err == 0.0, f"{name}: expected exact zeros, max err {err}"
        else:
            zb = np.asarray(zero_bound, dtype=np.float64).ravel()
            worst = np.max(np.abs(got) - zb)
            assert worst <= 0.0, f"{name}: expected zeros within the fp32 rounding bound, " \
                                 f"exceeded by {worst:.3e}"
        return {"cos": 1.0, "maxabs_rel": 0.0}
    cos = float(got @ ref / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    assert cos > cos_min, f"{name}: cos {cos:.6f} <= {cos_min}"
    assert err <= rel * scale, f"{name}: max abs err {err:.3e} > {rel} * {scale:.3e}"
    return {"cos": cos, "maxabs_rel": err / scale}


class Case:
    """One problem: seeded inputs, oracle O/lse (the backward's inputs) and device copies."""

    def __init__(self, inp: dict, device="cuda"):
        self.inp = inp
        self.T, self.H, self.D = inp["q"].shape
        self.N = inp["kv"].shape[0]
        self.K = inp["topk"].shape[1]
        self.scale = inp["scale"]
        self.r_chunk = inp.get("r_chunk", self.K)
        o_bits, lse32, _, _ = oracle.fwd_inputs(inp)
        self.o_bits, self.lse32 = o_bits, lse32
        # float64 views for the oracle
        self.q64 = oracle.bf16_to_f64(inp["q"])
        self.kv64 = oracle.bf16_to_f64(inp["kv"])
        self.do64 = oracle.bf16_to_f64(inp["do"])
        self.o64 = oracle.bf16_to_f64(o_bits)
        self.lse64 = lse32.astype(np.float64)
        self.sink64 = None if inp["sink"] is None else inp["sink"].astype(np.float64)
        # device copies
        self.q = bf16_dev(inp["q"], device)
        self.kv = bf16_dev(inp["kv"], device)
        self.do = bf16_dev(inp["do"], device)
        self.o = bf16_dev(o_bits, device)
        self.lse = torch.from_numpy(lse32).to(device)
        self.topk = torch.from_numpy(inp["topk"]).to(device)
        self.sink = None if inp["sink"] is None else torch.from_numpy(inp["sink"]).to(device)

    # ---------------------------------------------------------------- oracle
    def ref_full(self):
        return oracle.bwd(self.q64, self.kv64, self.do64, self.o64, self.lse64,
                          self.inp["topk"], self.sink64, self.scale)

    def ref_dq(self, tokens):
        return oracle.dq_tokens(self.q64, self.kv64, self.do64, self.o64, self.lse64,
                                self.inp["topk"], self.scale, tokens)

    def ref_dkv(self, rows):
        return oracle.dkv_rows(self.q64, self.kv64, self.do64, self.o64, self.lse64,
                               self.inp["topk"], self.scale, rows)

    def dq_zero_bound(self):
        """Elementwise bound on the GPU's dq where the exact dq is zero: topk = 1
        and no sink, so P = 1 and dS = P (dP - delta) with dP == delta exactly.

        The GPU forms dP (tensor-core accumulation) and delta (CUDA cores) as
        fp32 sums of the same 512 products dO[t,h,d] * kv[j,d] (exact in fp32)
        in different orders; each sum is within gamma_511 * sum_d |dO * kv| of
        the exact value (gamma_n = n u / (1 - n u), u = FP32_U). The kernel
        forms scale * dS = P * fma(dP, scale, -fl(scale * delta)): rounding
        scale * delta and the fma result adds at most 2 u * scale * |delta|
        <= 2 u * scale * sum_d |dO * kv| (|delta| = |sum_d dO * kv| here). Then
        scale * dS is rounded to bf16 (factor 1 + 2^-8), multiplied by kv[j, d]
        and the product rounded to bf16 again (1 + 2^-8); P itself is within
        1e-3 of 1 (P = exp(s - lse) with lse the fp32 rounding of s).
        """
        K = self.inp["topk"].shape[1]
        if K != 1 or self.sink64 is not None:
            raise ValueError("dq is identically zero only for topk = 1 without a sink")
        n = self.D - 1
        gamma = n * FP32_U / (1 - n * FP32_U)
        idx = self.inp["topk"][:, 0]
        bound = np.zeros((self.T, self.H, self.D))
        ok = idx >= 0
        kvr = self.kv64[np.where(ok, idx, 0)]                         # [T, D]
        s_abs = np.abs(self.do64 * kvr[:, None, :]).sum(axis=2)      # [T, H]
        diff = (2 * gamma + 2 * FP32_U) * s_abs                      # |dP - delta| on the GPU
        f = 1.001 * (1 + 2.0 ** -8) ** 2 * self.scale
        bound[ok] = (f * diff[:, :, None] * np.abs(kvr)[:, None, :])[ok]
        return bound

    def ref_dsink(self):
        return oracle.dsink(self.do64, self.o64, self.lse64, self.sink64)[0]


def custom_inputs(seed, T, H, K, N, sink=True, mask_p=0.2, dup=True, all_masked_rows=(),
                  r_chunk=0):
    """Small random problems with -1 slots, duplicate indices and fully masked rows."""
    rng = np.random.default_rng(seed)
    D = W.D_HEAD
    topk = rng.integers(0, N, size=(T, K)).astype(np.int32)
    if dup and T > 0 and K > 1:
        topk[0, 1] = topk[0, 0]
    if mask_p > 0:
        topk[rng.random((T, K)) < mask_p] = -1
    for t in all_masked_rows:
        topk[t, :] = -1
    return {
        "q": W.f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32)),
        "kv": W.f32_to_bf16_bits(rng.standard_normal((N, D), dtype=np.float32)),
        "do": W.f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32)),
        "sink": rng.standard_normal(H, dtype=np.float32) if sink else None,
        "topk": topk, "scale": float(1 / np.sqrt(D)), "r_chunk": r_chunk or K,
    }
