"""token_sparse_mla_gb300: token-sparse MLA attention forward for GB300 (sm_103a).

The work runs in the CUDA kernels of libsparse_mla.so; this module only
marshals torch tensors into the library's C ABI (include/sparse_mla.h).  There
is no fallback: if the library is missing or the tensors are not on a CUDA
device, the calls raise.

    out, lse = sparse_mla_fwd(q, kv_cache, indices, scale)

q [T, h, 576] bf16, kv_cache [num_slots, 576] bf16 (or [num_slots, 656] uint8
fp8 rows), indices [T, topk] int32 (-1 = invalid), h in {8, 16, 32, 64};
returns out [T, h, 512] bf16 and lse [T, h] fp32.  sparse_mla_merge combines
the (out, lse) of lists split into parts (the DCP merge); sparse_mla_v_up applies the
per-head value up-projection to out on the tensor cores; sparse_mla_topk builds the
index lists from per-position scores; sparse_mla_scatter_mask and sparse_mla_masked_mha are
the masked dense route for short prefills (the lists as a bit mask, then dense MHA over per-head
K and V under that mask).
"""

from ._binding import (  # noqa: F401
    KV_FORMATS,
    SparseMLAError,
    host_io_layout,
    host_io_views,
    host_workspace_bytes,
    launch_info,
    lib_path,
    library,
    sparse_mla_fwd,
    sparse_mla_fwd_host,
    sparse_mla_fwd_host_packed,
    sparse_mla_fwd_noalloc,
    sparse_mla_masked_mha,
    sparse_mla_merge,
    sparse_mla_scatter_mask,
    sparse_mla_topk,
    sparse_mla_v_up,
    sync_status,
    version,
)

__all__ = [
    "KV_FORMATS",
    "SparseMLAError",
    "host_io_layout",
    "host_io_views",
    "host_workspace_bytes",
    "launch_info",
    "lib_path",
    "library",
    "sparse_mla_fwd",
    "sparse_mla_fwd_host",
    "sparse_mla_fwd_host_packed",
    "sparse_mla_fwd_noalloc",
    "sparse_mla_masked_mha",
    "sparse_mla_merge",
    "sparse_mla_scatter_mask",
    "sparse_mla_topk",
    "sparse_mla_v_up",
    "sync_status",
    "version",
]
