"""Paged chunked-prefill attention for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of ``libpcp.so`` (declared in
``include/pcp.h``).  Every step of the path runs in the library's CUDA
kernels; this module only checks tensors, allocates outputs and workspace
with PyTorch, and passes raw pointers and the current CUDA stream.  There is
no CPU or PyTorch fallback: if the library is missing, importing the compute
functions raises.

Functions (same names as the C entry points, without the ``pcp_`` prefix):

* ``compute_out_cache_loc`` -- slots of a step's new tokens (int64)
* ``kv_append``             -- scatter the chunk's K/V into the page pools
* ``kv_append_paged``       -- slot mapping and KV append in one kernel
* ``copy_page_slots``       -- copy-on-write of shared pages
* ``paged_extend_attn``     -- extend attention, returns ``(out, lse)``
* ``workspace_size``        -- bytes of scratch a call needs
* ``Pager``                 -- host page pool and chunk planner of a serving step
"""
from ._binding import (  # noqa: F401
    Pager,
    PCPError,
    Status,
    compute_out_cache_loc,
    copy_page_slots,
    kv_append,
    kv_append_paged,
    lib,
    library_path,
    paged_extend_attn,
    read_error,
    workspace_size,
)

__all__ = [
    "Pager", "PCPError", "Status", "compute_out_cache_loc", "copy_page_slots", "kv_append",
    "kv_append_paged", "lib", "library_path", "paged_extend_attn", "read_error", "workspace_size",
]
