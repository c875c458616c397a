"""Torch-facing wrappers of the C ABI (marshalling only).

Every function takes CUDA tensors, checks dtypes / shapes / contiguity on the
host (the aiter page's wrapper checks, plus the dtype and lse-shape checks its
review asked for), passes raw device pointers and the current CUDA stream to
libsmla.so, and returns the outputs. All arithmetic runs in the library's
kernels. Nothing here falls back to PyTorch or the CPU: if libsmla.so is
missing or the device is not sm_103, the call raises.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import SmlaDims, SMLA_OP_BWD, SMLA_OP_BWD_HOST, SMLA_OP_CSR, SMLA_OP_FWD

D_HEAD = 512


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_dims(T: int, H: int, topk: int, num_kv: int, r_chunk: int = 0,
              scale: Optional[float] = None, D: int = D_HEAD) -> SmlaDims:
    return SmlaDims(T=T, H=H, D=D, topk=topk, num_kv=num_kv, r_chunk=r_chunk or 0,
                    scale=0.0 if scale is None else float(scale))


def workspace_size(op: int, dims: SmlaDims) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.load().smla_workspace_size(op, ctypes.byref(dims), ctypes.byref(n)),
               "smla_workspace_size")
    return int(n.value)


class Workspace:
    """A reusable device workspace (grown on demand, never shrunk)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


def device_status(workspace: torch.Tensor) -> int:
    """Sync the current stream and read the device status word of `workspace`."""
    st = ctypes.c_int(0)
    _lib.check(_lib.load().smla_get_device_status(_ptr(workspace), _stream(workspace.device),
                                                  ctypes.byref(st)), "smla_get_device_status")
    return int(st.value)


def sparse_mla_fwd(q: torch.Tensor, kv: torch.Tensor, topk: torch.Tensor,
                   sink: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                   workspace: Optional[Workspace] = None, check_status: bool = True,
                   out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None
                   ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Forward: (o [T,H,512] bf16, lse [T,H] fp32, sink-inclusive, natural log).

    `out` = (o, lse) writes into caller-owned tensors of those shapes."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kv, "kv", torch.bfloat16, 2)
    _need(topk, "topk", torch.int32, 2)
    T, H, D = q.shape
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        if sink.shape[0] != H:
            raise ValueError("sink must have shape [H]")
    if kv.shape[1] != D or topk.shape[0] != T:
        raise ValueError("shape mismatch between q, kv and topk")
    dims = make_dims(T, H, topk.shape[1], kv.shape[0], 0, scale, D)
    ws = (workspace or Workspace(q.device)).get(workspace_size(SMLA_OP_FWD, dims))
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
        _need(o, "o", torch.bfloat16, 3)
        _need(lse, "lse", torch.float32, 2)
        if tuple(o.shape) != (T, H, D) or tuple(lse.shape) != (T, H):
            raise ValueError("out must be (o [T,H,D], lse [T,H])")
    _lib.check(_lib.load().smla_fwd(_ptr(q), _ptr(kv), _ptr(topk), _ptr(sink), _ptr(o), _ptr(lse),
                                    ctypes.byref(dims), _ptr(ws), ws.numel(), _stream(q.device)),
               "smla_fwd")
    if check_status:
        st = device_status(ws)
        if st != _lib.SMLA_OK:
            raise _lib.SmlaError(st, "smla_fwd (device)")
    return o, lse


def sparse_mla_bwd(q: torch.Tensor, kv: torch.Tensor, do: torch.Tensor, o: torch.Tensor,
                   lse: torch.Tensor, topk: torch.Tensor, sink: Optional[torch.Tensor] = None,
                   scale: Optional[float] = None, r_chunk: Optional[int] = None,
                   workspace: Optional[Workspace] = None, out=None, check_status: bool = True):
    """Backward: (dq [T,H,512] bf16, dkv [num_kv,512] bf16, d_sink [H] fp32 or None).

    ``out`` may pass preallocated (dq, dkv, d_sink). With ``check_status`` the
    call synchronizes and raises if a kernel met an out-of-range index.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(kv, "kv", torch.bfloat16, 2)
    _need(do, "do", torch.bfloat16, 3)
    _need(o, "o", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    _need(topk, "topk", torch.int32, 2)
    T, H, D = q.shape
    if do.shape != q.shape or o.shape != q.shape:
        raise ValueError("do and o must have the shape of q")
    if tuple(lse.shape) != (T, H):
        raise ValueError("lse must have shape [T, H]")
    if kv.shape[1] != D or topk.shape[0] != T:
        raise ValueError("shape mismatch between q, kv and topk")
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        if sink.shape[0] != H:
            raise ValueError("sink must have shape [H]")
    for name, t in (("kv", kv), ("do", do), ("o", o), ("lse", lse), ("topk", topk), ("sink", sink)):
        if t is not None and t.device != q.device:
            raise ValueError(f"{name} must be on {q.device}, got {t.device}")
    dims = make_dims(T, H, topk.shape[1], kv.shape[0], r_chunk or 0, scale, D)
    ws = (workspace or Workspace(q.device)).get(workspace_size(SMLA_OP_BWD, dims))
    if out is None:
        dq = torch.empty_like(q)
        dkv = torch.empty_like(kv)
        d_sink = None if sink is None else torch.empty(H, dtype=torch.float32, device=q.device)
    else:
        dq, dkv, d_sink = out
        _need(dq, "dq", torch.bfloat16, 3)
        _need(dkv, "dkv", torch.bfloat16, 2)
        if tuple(dq.shape) != (T, H, D) or tuple(dkv.shape) != tuple(kv.shape):
            raise ValueError("out must be (dq [T,H,D], dkv [num_kv,D], d_sink [H] or None)")
        if (d_sink is None) != (sink is None):
            raise ValueError("out's d_sink must be given exactly when sink is given")
        if d_sink is not None:
            _need(d_sink, "d_sink", torch.float32, 1)
            if d_sink.shape[0] != H:
                raise ValueError("d_sink must have shape [H]")
        for name, t in (("dq", dq), ("dkv", dkv), ("d_sink", d_sink)):
            if t is not None and t.device != q.device:
                raise ValueError(f"{name} must be on {q.device}, got {t.device}")
    _lib.check(_lib.load().smla_bwd(_ptr(q), _ptr(kv), _ptr(do), _ptr(o), _ptr(lse), _ptr(topk),
                                    _ptr(sink), _ptr(dq), _ptr(dkv), _ptr(d_sink),
                                    ctypes.byref(dims), _ptr(ws), ws.numel(), _stream(q.device)),
               "smla_bwd")
    if check_status:
        st = device_status(ws)
        if st != _lib.SMLA_OK:
            raise _lib.SmlaError(st, "smla_bwd (device)")
    return dq, dkv, d_sink


def sparse_mla_bwd_partial(q: torch.Tensor, kv: torch.Tensor, do: torch.Tensor, o: torch.Tensor,
                           lse: torch.Tensor, topk: torch.Tensor, sink: Optional[torch.Tensor] = None,
                           scale: Optional[float] = None, r_chunk: Optional[int] = None,
                           workspace: Optional[Workspace] = None, check_status: bool = True):
    """One rank's share of a token-sharded backward (smla_bwd_partial).

    q, do, o, lse, topk hold this rank's tokens; kv (and sink) are the full
    tensors. Returns (dq [T,H,512] bf16, dkv_partial [num_kv,512] fp32,
    d_sink_partial [H] fp32 or None): the kv and sink gradients summed over
    this rank's tokens only, unrounded.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(kv, "kv", torch.bfloat16, 2)
    _need(do, "do", torch.bfloat16, 3)
    _need(o, "o", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    _need(topk, "topk", torch.int32, 2)
    T, H, D = q.shape
    if do.shape != q.shape or o.shape != q.shape:
        raise ValueError("do and o must have the shape of q")
    if tuple(lse.shape) != (T, H):
        raise ValueError("lse must have shape [T, H]")
    if kv.shape[1] != D or topk.shape[0] != T:
        raise ValueError("shape mismatch between q, kv and topk")
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        if sink.shape[0] != H:
            raise ValueError("sink must have shape [H]")
    for name, t in (("kv", kv), ("do", do), ("o", o), ("lse", lse), ("topk", topk), ("sink", sink)):
        if t is not None and t.device != q.device:
            raise ValueError(f"{name} must be on {q.device}, got {t.device}")
    dims = make_dims(T, H, topk.shape[1], kv.shape[0], r_chunk or 0, scale, D)
    ws = (workspace or Workspace(q.device)).get(workspace_size(SMLA_OP_BWD, dims))
    dq = torch.empty_like(q)
    dkv = torch.empty(kv.shape, dtype=torch.float32, device=q.device)
    d_sink = None if sink is None else torch.empty(H, dtype=torch.float32, device=q.device)
    _lib.check(_lib.load().smla_bwd_partial(_ptr(q), _ptr(kv), _ptr(do), _ptr(o), _ptr(lse),
                                            _ptr(topk), _ptr(sink), _ptr(dq), _ptr(dkv),
                                            _ptr(d_sink), ctypes.byref(dims), _ptr(ws), ws.numel(),
                                            _stream(q.device)),
               "smla_bwd_partial")
    if check_status:
        st = device_status(ws)
        if st != _lib.SMLA_OK:
            raise _lib.SmlaError(st, "smla_bwd_partial (device)")
    return dq, dkv, d_sink


def reduce_partials(partials: torch.Tensor, want_bf16: bool = True, want_f32: bool = False):
    """Ordered sum over the first dimension of partials [n_parts, n] fp32
    (smla_reduce_partials): parts added in index order, in fp32.
    Returns (sum rounded to bf16 or None, fp32 sum or None)."""
    _need(partials, "partials", torch.float32, 2)
    if not (want_bf16 or want_f32):
        raise ValueError("ask for a bf16 or an fp32 result")
    n_parts, n = partials.shape
    out_b = torch.empty(n, dtype=torch.bfloat16, device=partials.device) if want_bf16 else None
    out_f = torch.empty(n, dtype=torch.float32, device=partials.device) if want_f32 else None
    _lib.check(_lib.load().smla_reduce_partials(_ptr(partials), int(n_parts), int(n), _ptr(out_b),
                                                _ptr(out_f), _stream(partials.device)),
               "smla_reduce_partials")
    return out_b, out_f


def _need_host(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def sparse_mla_bwd_host(q: torch.Tensor, kv: torch.Tensor, do: torch.Tensor, o: torch.Tensor,
                        lse: torch.Tensor, topk: torch.Tensor, sink: Optional[torch.Tensor] = None,
                        scale: Optional[float] = None, r_chunk: Optional[int] = None,
                        workspace: Optional[Workspace] = None, out=None, device=None,
                        synchronize: bool = True, check_status: bool = True):
    """Backward with host (CPU) inputs and outputs, through smla_bwd_host.

    The library copies the inputs to the device in token chunks, overlapping
    the copies with the compute, and copies dq, dkv and d_sink back. Pinned
    host tensors (``tensor.pin_memory()``) let the copies run asynchronously.
    ``out`` may pass preallocated host (dq, dkv, d_sink). With ``synchronize``
    the call waits for the results (and, with ``check_status``, raises if a
    kernel met an out-of-range index); without it the results are valid once
    the current CUDA stream of ``device`` has completed.
    """
    _need_host(q, "q", torch.bfloat16, 3)
    _need_host(kv, "kv", torch.bfloat16, 2)
    _need_host(do, "do", torch.bfloat16, 3)
    _need_host(o, "o", torch.bfloat16, 3)
    _need_host(lse, "lse", torch.float32, 2)
    _need_host(topk, "topk", torch.int32, 2)
    T, H, D = q.shape
    if do.shape != q.shape or o.shape != q.shape:
        raise ValueError("do and o must have the shape of q")
    if tuple(lse.shape) != (T, H):
        raise ValueError("lse must have shape [T, H]")
    if kv.shape[1] != D or topk.shape[0] != T:
        raise ValueError("shape mismatch between q, kv and topk")
    if sink is not None:
        _need_host(sink, "sink", torch.float32, 1)
        if sink.shape[0] != H:
            raise ValueError("sink must have shape [H]")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    dims = make_dims(T, H, topk.shape[1], kv.shape[0], r_chunk or 0, scale, D)
    ws = (workspace or Workspace(dev)).get(workspace_size(SMLA_OP_BWD_HOST, dims))
    if out is None:
        pin = q.is_pinned()
        dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
        dkv = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=pin)
        d_sink = None if sink is None else torch.empty(H, dtype=torch.float32, pin_memory=pin)
    else:
        dq, dkv, d_sink = out
        _need_host(dq, "dq", torch.bfloat16, 3)
        _need_host(dkv, "dkv", torch.bfloat16, 2)
        if d_sink is not None:
            _need_host(d_sink, "d_sink", torch.float32, 1)
    _lib.check(_lib.load().smla_bwd_host(_ptr(q), _ptr(kv), _ptr(do), _ptr(o), _ptr(lse), _ptr(topk),
                                         _ptr(sink), _ptr(dq), _ptr(dkv), _ptr(d_sink),
                                         ctypes.byref(dims), _ptr(ws), ws.numel(), _stream(dev)),
               "smla_bwd_host")
    if synchronize:
        torch.cuda.current_stream(dev).synchronize()
        if check_status:
            st = device_status(ws)
            if st != _lib.SMLA_OK:
                raise _lib.SmlaError(st, "smla_bwd_host (device)")
    return dq, dkv, d_sink


def csr_build(topk: torch.Tensor, num_kv: int, r0: int = 0, r_len: Optional[int] = None,
              workspace: Optional[Workspace] = None, check_status: bool = True):
    """Inverted top-k CSR over ranks [r0, r0+r_len): (row_ptr [num_kv+1], col [nnz]) int32."""
    _need(topk, "topk", torch.int32, 2)
    T, W = topk.shape
    R = W - r0 if r_len is None else r_len
    dims = make_dims(T, 16, W, num_kv, R)
    ws = (workspace or Workspace(topk.device)).get(workspace_size(SMLA_OP_CSR, dims))
    row_ptr = torch.empty(num_kv + 1, dtype=torch.int32, device=topk.device)
    col = torch.empty(max(T * R, 4), dtype=torch.int32, device=topk.device)
    _lib.check(_lib.load().smla_csr_build(_ptr(topk), T, W, r0, R, num_kv, _ptr(row_ptr), _ptr(col),
                                          _ptr(ws), ws.numel(), _stream(topk.device)),
               "smla_csr_build")
    if check_status:
        st = device_status(ws)
        if st != _lib.SMLA_OK:
            raise _lib.SmlaError(st, "smla_csr_build (device)")
    nnz = int(row_ptr[-1].item())
    return row_ptr, col[:nnz]


def default_scale(D: int = D_HEAD) -> float:
    return 1.0 / math.sqrt(D)
