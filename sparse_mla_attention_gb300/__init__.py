"""GB300-native (sm_103a) sparse MLA attention: forward for inputs, training backward.

The compute runs in ``libsmla.so`` (hand-written CUDA kernels behind the C ABI
of ``include/smla.h``). This package only marshals torch tensors into that
ABI (``api``), builds the library (``build``), draws seeded synthetic
inputs (``workloads``) and runs a token-sharded backward over several GPUs
(``sharded``: torch.distributed moves the partials, the library adds them).
"""

from .api import (Workspace, csr_build, default_scale, device_status, make_dims, reduce_partials,
                  sparse_mla_bwd, sparse_mla_bwd_host, sparse_mla_bwd_partial, sparse_mla_fwd,
                  workspace_size)
from ._lib import SmlaError

__all__ = ["Workspace", "csr_build", "default_scale", "device_status", "make_dims",
           "reduce_partials", "sparse_mla_bwd", "sparse_mla_bwd_host", "sparse_mla_bwd_partial",
           "sparse_mla_fwd", "workspace_size", "SmlaError"]
