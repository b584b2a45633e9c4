"""Chunkwise-parallel DeltaNet / Gated DeltaNet on one GB300 (sm_103a).

The computation lives in libgdn_gb300.so (C ABI, include/gdn.h); ``binding``
marshals torch tensors into it.  ``workloads`` holds the seeded synthetic
inputs.
"""
from . import workloads  # noqa: F401
from .binding import (  # noqa: F401
    DnShape, GdnError, backward, decode_step, dn_chunk_fwd, dn_device_status, dn_host_arena_size,
    dn_saved_size, dn_uses_fast_path, dn_workspace_size, forward, gdn_chunk_bwd, gdn_chunk_bwd_saved,
    gdn_chunk_fwd, gdn_chunk_fwd_host, gdn_chunk_fwd_noalloc, gdn_chunk_fwd_save, gdn_decode_step,
    make_shape, saved_supported,
)
