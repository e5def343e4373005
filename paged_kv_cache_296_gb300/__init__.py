"""GB300-native paged KV cache: reshape_and_cache and paged decode attention.

The compute lives in ``_lib/libpagedattn.so`` (hand-written CUDA for sm_103a,
C ABI in ``include/pa.h``); :mod:`.binding` marshals torch tensors into its
calls.  Build the library with :func:`build`.
"""

from .binding import (  # noqa: F401
    PagedAttentionError, kv_views, load, pa_check_tables, pa_decode, pa_decode_append,
    pa_decode_noalloc, pa_decode_partition_size, pa_prefill, pa_decode_workspace_size,
    pa_device_status, pa_gather_kv, pa_last_error, pa_reshape_and_cache, pa_version,
    alloc_workspace, dtype_code, BlockManager, OutOfBlocks, pa_copy_blocks, SharedGroups,
    pa_decode_shared, pa_decode_append_shared, pa_decode_shared_workspace_size,
    pa_find_shared_prefixes,
)


def build(force=False):
    """Compile the CUDA library in-tree (nvcc, sm_103a) and return its path."""
    from .native_build import build as _build
    return _build(force=force)
