"""Python binding of libpagedattn.so: argument marshalling only.

Every function has the name of the C entry point it calls (see include/pa.h)
and turns torch tensors into the pointers, sizes and dtype codes that entry
point takes; all computation runs in the library's CUDA kernels on the
tensors' device and the current torch stream.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""

import ctypes
import os

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpagedattn.so")

PA_F16, PA_BF16, PA_E4M3, PA_F32 = 0, 1, 2, 3
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_WORKSPACE", 4: "PA_ERR_CUDA", 5: "PA_ERR_BAD_INDEX",
                6: "PA_ERR_OUT_OF_BLOCKS"}

#: Every function include/pa.h declares, with (restype, argtypes).
_P, _I, _I64, _F, _SZ, _U32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_size_t, ctypes.c_uint32)
SIGNATURES = {
    "pa_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _I, _I, _F, _P]),
    "pa_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _F, _I,
                       _P, _SZ, _P]),
    "pa_decode_append": (_I, [_P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                              _F, _I, _I, _F, _I, _P, _SZ, _P]),
    "pa_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                               _F, _I, _P]),
    "pa_decode_shared": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _F,
                              _P, _P, _P, _I, _P, _SZ, _P]),
    "pa_decode_append_shared": (_I, [_P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I, _I, _I, _I,
                                     _I, _I, _I, _F, _I, _I, _F, _P, _P, _P, _I, _P, _SZ, _P]),
    "pa_decode_shared_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_find_shared_prefixes": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "pa_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                        _F, _P]),
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_decode_partition_size": (_I, [_I, _I, _I, _I, _I]),
    "pa_gather_kv": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "pa_check_tables": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P]),
    "pa_device_status": (_U32, [_I]),
    "pa_bm_create": (_P, [ctypes.c_int32, ctypes.c_int32]),
    "pa_bm_destroy": (None, [_P]),
    "pa_bm_num_free": (ctypes.c_int32, [_P]),
    "pa_bm_ref_count": (ctypes.c_int32, [_P, ctypes.c_int32]),
    "pa_bm_allocate": (_I, [_P, _I64, _I64]),
    "pa_bm_append_batch": (_I, [_P, _P, _P, ctypes.c_int32, _P, _P, _P]),
    "pa_bm_append": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "pa_bm_fork": (_I, [_P, _I64, _I64]),
    "pa_bm_allocate_cached": (_I, [_P, _I64, _P, _I64, _P]),
    "pa_bm_register": (_I, [_P, _I64, _P, _I64]),
    "pa_bm_free": (_I, [_P, _I64]),
    "pa_bm_block_tables": (_I, [_P, _P, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "pa_copy_blocks": (_I, [_P, _P, _I64, ctypes.c_int32, _I64, _P]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (_I, []),
}


class PagedAttentionError(RuntimeError):
    """A library call returned a non-zero pa_status."""

    def __init__(self, fn, status, message):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path=LIB_PATH):
    """Load the library (once) and declare its signatures.  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn, status):
    if status != 0:
        raise PagedAttentionError(fn, status, load().pa_last_error().decode())


def dtype_code(dt):
    if dt == torch.float16:
        return PA_F16
    if dt == torch.bfloat16:
        return PA_BF16
    if dt in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return PA_E4M3
    if dt == torch.float32:
        return PA_F32
    raise ValueError(f"unsupported dtype {dt}")


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def kv_views(pool):
    """K and V views ``[num_blocks, 16, Hkv, D]`` of a pool ``[num_blocks, 16, 2, Hkv, D]``."""
    if pool.dim() != 5 or pool.shape[2] != 2 or not pool.is_contiguous():
        raise ValueError("pool must be a contiguous [num_blocks, block_size, 2, Hkv, D] tensor")
    return pool[:, :, 0], pool[:, :, 1]


def _cache_geometry(k_cache, v_cache):
    """(num_blocks, block_size, Hkv, D) of K/V views, checking the pool strides."""
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must be [num_blocks, block_size, Hkv, D] views")
    nb, bs, hkv, d = k_cache.shape
    want = (bs * 2 * hkv * d, 2 * hkv * d, d, 1)
    if tuple(k_cache.stride()) != want or tuple(v_cache.stride()) != want:
        raise ValueError("k_cache/v_cache must be the c=0/c=1 views of a "
                         "[num_blocks, block_size, 2, Hkv, D] pool")
    return nb, bs, hkv, d


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, kv_scale=1.0):
    """Write ``k``/``v`` ``[n_tokens, Hkv, D]`` into the pool at ``slot_mapping`` (int64)."""
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    if k.shape != v.shape or k.dim() != 3 or k.stride() != v.stride() or k.stride(1) != d \
            or k.stride(2) != 1:
        raise ValueError("k and v must be [n_tokens, Hkv, D] with unit inner strides")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 tensor")
    lib = load()
    st = lib.pa_reshape_and_cache(
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), k.shape[0],
        k.stride(0), nb, hkv, d, bs, dtype_code(k.dtype), dtype_code(k_cache.dtype),
        float(kv_scale), _stream(k_cache))
    _check("pa_reshape_and_cache", st)


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, max_blocks_per_seq,
                             block_size=16, partition_size=0):
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                               max_blocks_per_seq, block_size, partition_size))


def pa_decode_partition_size(num_seqs, num_kv_heads, max_blocks_per_seq, block_size=16,
                             partition_size=0):
    return int(load().pa_decode_partition_size(num_seqs, num_kv_heads, max_blocks_per_seq,
                                               block_size, partition_size))


def alloc_workspace(nbytes, device):
    """Device scratch for pa_decode's split-KV partials (256-byte aligned), or None."""
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, kv_scale=1.0,
              partition_size=0, workspace=None):
    """Paged decode attention into ``out`` ``[B, Hq, D]``.

    ``workspace``: a uint8 device tensor of at least ``pa_decode_workspace_size``
    bytes; allocated here when omitted.
    """
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables and context_lens must be contiguous int32 tensors")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks], context_lens [B]")
    mb = block_tables.shape[1]
    need = pa_decode_workspace_size(B, hq, hkv, d, mb, bs, partition_size)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, mb, nb, hq, hkv, d, bs, float(scale), dtype_code(q.dtype), dtype_code(k_cache.dtype),
        float(kv_scale), int(partition_size), _ptr(workspace), wbytes, _stream(q))
    _check("pa_decode", st)


def pa_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
               max_query_len, scale, kv_scale=1.0):
    """Causal paged prefill into ``out`` ``[T, Hq, D]`` (rows of ``q``).

    ``query_start_loc``: int32 ``[B + 1]``; sequence i's queries are rows
    ``query_start_loc[i] .. query_start_loc[i+1]-1``, its last tokens.  The
    cache is of q's dtype, or uint8 E4M3 codes with values ``code * kv_scale``.
    """
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    T, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [T, Hq, D] tensors")
    B = context_lens.shape[0]
    for t in (block_tables, context_lens, query_start_loc):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("block_tables, context_lens and query_start_loc must be contiguous int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or query_start_loc.shape != (B + 1,):
        raise ValueError("block_tables must be [B, max_blocks], query_start_loc [B + 1]")
    if k_cache.dtype != q.dtype and k_cache.dtype != torch.uint8:
        raise ValueError("pa_prefill reads a cache of q's dtype or of E4M3 codes (uint8)")
    st = load().pa_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), B, int(max_query_len), block_tables.shape[1], nb, hq, hkv, d, bs,
        float(scale), dtype_code(q.dtype), dtype_code(k_cache.dtype), float(kv_scale), _stream(q))
    _check("pa_prefill", st)


def pa_decode_append(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                     context_lens, scale, kv_scale=1.0, partition_size=0, workspace=None):
    """Write each sequence's new token (``k_new``/``v_new`` ``[B, Hkv, D]``) and decode, in one launch."""
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    if k_new.shape != (B, hkv, d) or v_new.shape != k_new.shape or k_new.stride() != v_new.stride() \
            or k_new.stride(1) != d or k_new.stride(2) != 1 or k_new.dtype != q.dtype \
            or v_new.dtype != q.dtype:
        raise ValueError("k_new and v_new must be [B, Hkv, D] of q's dtype with unit inner strides")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous() \
            or slot_mapping.shape != (B,):
        raise ValueError("slot_mapping must be a contiguous int64 [B] tensor")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables and context_lens must be contiguous int32 tensors")
    mb = block_tables.shape[1]
    need = pa_decode_workspace_size(B, hq, hkv, d, mb, bs, partition_size)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_decode_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.stride(0),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, mb, nb, hq, hkv,
        d, bs, float(scale), dtype_code(q.dtype), dtype_code(k_cache.dtype), float(kv_scale),
        int(partition_size), _ptr(workspace), wbytes, _stream(q))
    _check("pa_decode_append", st)


def pa_decode_shared_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                    max_blocks_per_seq, block_size=16, num_groups=0):
    return int(load().pa_decode_shared_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                      head_size, max_blocks_per_seq, block_size,
                                                      num_groups))


class SharedGroups:
    """pa_decode_shared's group arrays (device int32 tensors, CSR over sequences)."""

    def __init__(self, offsets, seqs, blocks):
        self.offsets, self.seqs, self.blocks = offsets, seqs, blocks

    @property
    def num_groups(self):
        return self.offsets.numel() - 1

    def to(self, device):
        return SharedGroups(self.offsets.to(device), self.seqs.to(device), self.blocks.to(device))


def pa_find_shared_prefixes(block_tables, context_lens, num_q_heads, num_kv_heads, min_blocks=1,
                            block_size=16):
    """Groups of sequences whose (host) tables start with the same blocks, as
    :class:`SharedGroups` of CPU tensors (``.to(device)`` for the decode)."""
    bt = block_tables.to("cpu", torch.int32).contiguous()
    cl = context_lens.to("cpu", torch.int32).contiguous()
    B = cl.shape[0]
    if bt.dim() != 2 or bt.shape[0] != B:
        raise ValueError("block_tables must be [B, max_blocks], context_lens [B]")
    offs = torch.zeros(B + 1, dtype=torch.int32)
    seqs = torch.zeros(max(B, 1), dtype=torch.int32)
    blks = torch.zeros(max(B, 1), dtype=torch.int32)
    ng = ctypes.c_int32(0)
    st = load().pa_find_shared_prefixes(_ptr(bt), _ptr(cl), B, bt.shape[1], block_size,
                                        num_q_heads, num_kv_heads, int(min_blocks), _ptr(offs),
                                        _ptr(seqs), _ptr(blks), ctypes.byref(ng))
    _check("pa_find_shared_prefixes", st)
    n = ng.value
    nm = int(offs[n])
    return SharedGroups(offs[:n + 1].clone(), seqs[:max(nm, 1)].clone(), blks[:max(n, 1)].clone())


def _shared_args(groups):
    if groups.offsets.dtype != torch.int32 or groups.seqs.dtype != torch.int32 \
            or groups.blocks.dtype != torch.int32:
        raise ValueError("group arrays must be int32")
    return _ptr(groups.offsets), _ptr(groups.seqs), _ptr(groups.blocks), groups.num_groups


def pa_decode_shared(out, q, k_cache, v_cache, block_tables, context_lens, scale, groups,
                     kv_scale=1.0, workspace=None):
    """pa_decode with shared-prefix ``groups`` (:class:`SharedGroups` on q's device)."""
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables and context_lens must be contiguous int32 tensors")
    mb = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(
            pa_decode_shared_workspace_size(B, hq, hkv, d, mb, bs, groups.num_groups), q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_decode_shared(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, mb, nb, hq, hkv, d, bs, float(scale), dtype_code(q.dtype), dtype_code(k_cache.dtype),
        float(kv_scale), *_shared_args(groups), _ptr(workspace), wbytes, _stream(q))
    _check("pa_decode_shared", st)


def pa_decode_append_shared(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                            context_lens, scale, groups, kv_scale=1.0, workspace=None):
    """pa_decode_append with shared-prefix ``groups``: write each new token, then decode."""
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    if k_new.shape != (B, hkv, d) or v_new.shape != k_new.shape or k_new.stride() != v_new.stride() \
            or k_new.stride(1) != d or k_new.stride(2) != 1 or k_new.dtype != q.dtype \
            or v_new.dtype != q.dtype:
        raise ValueError("k_new and v_new must be [B, Hkv, D] of q's dtype with unit inner strides")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous() \
            or slot_mapping.shape != (B,):
        raise ValueError("slot_mapping must be a contiguous int64 [B] tensor")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables and context_lens must be contiguous int32 tensors")
    mb = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(
            pa_decode_shared_workspace_size(B, hq, hkv, d, mb, bs, groups.num_groups), q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_decode_append_shared(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.stride(0),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, mb, nb, hq, hkv,
        d, bs, float(scale), dtype_code(q.dtype), dtype_code(k_cache.dtype), float(kv_scale),
        *_shared_args(groups), _ptr(workspace), wbytes, _stream(q))
    _check("pa_decode_append_shared", st)


#: Bytes of the library's fixed split-KV scratch used by pa_decode_noalloc.
DECODE_NOALLOC_SCRATCH_BYTES = 64 << 20


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale, kv_scale=1.0,
                      partition_size=0):
    """Paged decode with the library's own fixed scratch: no workspace, no allocation.

    For callers that cannot allocate device memory.  Calls on one device share
    that scratch, so calls that overlap on the GPU race; keep them on one stream.
    """
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, hq, dq = q.shape
    if dq != d or out.shape != q.shape or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables and context_lens must be contiguous int32 tensors")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks], context_lens [B]")
    st = load().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, block_tables.shape[1], nb, hq, hkv, d, bs, float(scale), dtype_code(q.dtype),
        dtype_code(k_cache.dtype), float(kv_scale), int(partition_size), _stream(q))
    _check("pa_decode_noalloc", st)


def pa_gather_kv(k_out, v_out, k_cache, v_cache, block_tables, context_lens, cu_seqlens):
    """Copy each sequence's cached K/V rows, in token order, into ``k_out``/``v_out``."""
    nb, bs, hkv, d = _cache_geometry(k_cache, v_cache)
    B, mb = block_tables.shape
    st = load().pa_gather_kv(
        _ptr(k_out), _ptr(v_out), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), _ptr(cu_seqlens), B, mb, nb, hkv, d, bs, dtype_code(k_cache.dtype),
        _stream(k_cache))
    _check("pa_gather_kv", st)


def pa_check_tables(block_tables, context_lens, slot_mapping, num_blocks, block_size=16):
    """Validate index arrays; returns the three counts (see include/pa.h)."""
    B, mb = block_tables.shape
    counts_dev = torch.zeros(3, dtype=torch.int32, device=block_tables.device)
    counts_host = (ctypes.c_int32 * 3)()
    n = 0 if slot_mapping is None else slot_mapping.numel()
    st = load().pa_check_tables(
        _ptr(block_tables), _ptr(context_lens), _ptr(slot_mapping) if n else ctypes.c_void_p(0),
        n, B, mb, num_blocks, block_size, _ptr(counts_dev), ctypes.cast(counts_host, ctypes.c_void_p),
        _stream(block_tables))
    counts = list(counts_host)
    if st not in (0, 5):
        _check("pa_check_tables", st)
    return counts


def pa_device_status(clear=True):
    return int(load().pa_device_status(1 if clear else 0))


def pa_last_error():
    return load().pa_last_error().decode()


def pa_version():
    return int(load().pa_version())


# ---------------------------------------------------------------- block manager

class OutOfBlocks(PagedAttentionError):
    """The block manager has too few free blocks (the call changed nothing)."""


class BlockManager:
    """The library's native block allocator (pa_bm_* in include/pa.h).

    Sequence ids are Python ints.  ``append`` returns the new tokens' slots
    (the slot_mapping of pa_reshape_and_cache) and the copy-on-write block
    pairs to copy first (pa_copy_blocks).
    """

    def __init__(self, num_blocks, block_size=16):
        self._lib = load()
        self._h = self._lib.pa_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise PagedAttentionError("pa_bm_create", 1, self._lib.pa_last_error().decode())
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pa_bm_destroy(h)

    def _check(self, fn, st):
        if st == 6:
            raise OutOfBlocks(fn, st, self._lib.pa_last_error().decode())
        _check(fn, st)

    def num_free(self):
        return self._lib.pa_bm_num_free(self._h)

    def ref_count(self, block):
        return self._lib.pa_bm_ref_count(self._h, int(block))

    def allocate(self, seq_id, num_tokens):
        self._check("pa_bm_allocate", self._lib.pa_bm_allocate(self._h, int(seq_id), int(num_tokens)))

    def append_batch(self, seq_ids, counts, as_arrays=False):
        """Reserve counts[i] tokens for seq_ids[i].

        Returns (slots, copies): lists, or with ``as_arrays`` an int64 NumPy
        array of slots and an int64 ``[n_copies, 2]`` array of pairs.
        """
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int64)
        n = ids.shape[0]
        total = int(cnt.sum()) if n else 0
        slots = np.empty(max(total, 1), dtype=np.int64)
        copies = np.empty((max(n, 1), 2), dtype=np.int64)
        ncopy = ctypes.c_int32(0)
        st = self._lib.pa_bm_append_batch(self._h, ids.ctypes.data, cnt.ctypes.data, n,
                                          slots.ctypes.data, copies.ctypes.data,
                                          ctypes.byref(ncopy))
        self._check("pa_bm_append_batch", st)
        slots, copies = slots[:total], copies[:ncopy.value]
        if as_arrays:
            return slots, copies
        return slots.tolist(), [tuple(c) for c in copies.tolist()]

    def append(self, seq_id, n):
        return self.append_batch([seq_id], [n])

    def allocate_cached(self, seq_id, tokens):
        """A new sequence for the prompt ``tokens`` (ints) with prefix caching;
        returns how many leading tokens are already cached."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = ctypes.c_int64(0)
        st = self._lib.pa_bm_allocate_cached(self._h, int(seq_id), toks.ctypes.data,
                                             toks.shape[0], ctypes.byref(cached))
        self._check("pa_bm_allocate_cached", st)
        return cached.value

    def register(self, seq_id, tokens):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        self._check("pa_bm_register",
                    self._lib.pa_bm_register(self._h, int(seq_id), toks.ctypes.data, toks.shape[0]))

    def fork(self, parent, child):
        self._check("pa_bm_fork", self._lib.pa_bm_fork(self._h, int(parent), int(child)))

    def free(self, seq_id):
        self._check("pa_bm_free", self._lib.pa_bm_free(self._h, int(seq_id)))

    def block_tables(self, seq_ids, width, out=None):
        """int32 tensors (tables [n, width] padded with -1, lengths [n]) on the CPU.

        ``out``: (tables, lens) to write instead of new tensors, e.g. pinned
        buffers a serving loop copies to the GPU each step; contiguous int32
        CPU tensors of at least [n, width] and [n] elements (rows beyond n are
        left as they are).
        """
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        if out is None:
            tables = torch.empty((n, width), dtype=torch.int32)
            lens = torch.empty((n,), dtype=torch.int32)
        else:
            tables, lens = out
            for t, need in ((tables, n * width), (lens, n)):
                if (t.dtype != torch.int32 or t.device.type != "cpu" or not t.is_contiguous()
                        or t.numel() < need):
                    raise ValueError("out must be contiguous int32 CPU tensors large enough "
                                     "for [n, width] and [n]")
            if tables.dim() != 2 or tables.shape[1] != width:
                raise ValueError("out tables must be [rows, width]")
        st = self._lib.pa_bm_block_tables(self._h, ids.ctypes.data, n, int(width),
                                          ctypes.c_void_p(tables.data_ptr()),
                                          ctypes.c_void_p(lens.data_ptr()))
        self._check("pa_bm_block_tables", st)
        return tables[:n], lens[:n]


def pa_copy_blocks(pool, pairs):
    """Copy whole physical blocks of ``pool`` ``[NB, BS, 2, Hkv, D]`` on its device:
    ``pairs`` int64 ``[n, 2]`` (src, dst) on the same device."""
    if not pool.is_contiguous() or pairs.dtype != torch.int64 or not pairs.is_contiguous():
        raise ValueError("pool must be contiguous and pairs a contiguous int64 [n, 2] tensor")
    nb = pool.shape[0]
    block_bytes = pool[0].numel() * pool.element_size()
    st = load().pa_copy_blocks(_ptr(pool), _ptr(pairs), int(pairs.shape[0]), nb, block_bytes,
                               _stream(pool))
    _check("pa_copy_blocks", st)
