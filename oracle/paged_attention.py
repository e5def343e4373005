"""Plain float64 definition of the paged-KV-cache decode hot path.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Slow on purpose: every
step is written the way the pages describe it, with NumPy as the only
library, so a reader can check it against the pages by eye.

Storage convention shared with the tests: every array that stands for GPU
memory holds raw element *bits* plus a dtype tag, because NumPy has no
bfloat16 or E4M3 type.

  ``"f16"``  -- IEEE binary16, stored as uint16 bits
  ``"bf16"`` -- bfloat16, stored as uint16 bits (the top half of a float32)
  ``"f32"``  -- IEEE binary32, stored as uint32 bits
  ``"e4m3"`` -- OCP E4M3, stored as uint8 codes

The KV pool is the pages' single preallocated tensor
``[num_blocks, block_size, 2, num_kv_heads, head_size]`` ("vLLM 部署深度指南",
section 代码层面理解, the ``kv_pool`` allocation); index 2 selects K (0) or V (1).
"""

import numpy as np

from . import e4m3

#: Storage dtype of each tag.
STORAGE = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32, "e4m3": np.uint8}


# --------------------------------------------------------------------------
# Element widening / narrowing (exact, except where a rounding rule is named)
# --------------------------------------------------------------------------

def widen(bits, dtype):
    """Exact float64 value of stored elements ``bits`` of type ``dtype``."""
    bits = np.asarray(bits)
    if dtype == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        # A bfloat16 is the upper 16 bits of the float32 with the same value.
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "e4m3":
        return e4m3.decode(bits)
    raise ValueError(f"unknown dtype {dtype!r}")


def narrow_f32(x):
    """Round float64 values to float32 (IEEE round-to-nearest-even), as float32."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fp8_quantise(src_bits, src_dtype, kv_scale):
    """fp8 KV write rule: ``e4m3_rn_sat(float32(x) / float32(kv_scale))``.

    The quotient is one IEEE float32 division (correctly rounded), then one
    rounding to E4M3 (nearest, ties to even, saturating at 448).  The pages fix
    only that the cache is fp8 ("vLLM 部署深度指南", 量化支持 table, FP8 row); the
    division-then-round order with a per-tensor scale is the plainest reading
    of a per-tensor-scaled fp8 cache.
    """
    x32 = narrow_f32(widen(src_bits, src_dtype))   # exact: every source type fits in f32
    s32 = np.float32(kv_scale)
    y32 = x32 / s32                                 # NumPy float32 division is IEEE-rounded
    return e4m3.encode(y32.astype(np.float64))


def fp8_dequantise(codes, kv_scale):
    """Value the fp8 cache stands for: ``decode(code) * kv_scale`` in float64."""
    return e4m3.decode(codes) * np.float64(np.float32(kv_scale))


# --------------------------------------------------------------------------
# Slot arithmetic and the block-table gather
# --------------------------------------------------------------------------

def blocks_needed(num_tokens, block_size):
    """Blocks a sequence of ``num_tokens`` tokens occupies: the ceiling of the ratio.

    "vLLM 部署深度指南", section 代码层面理解, ``allocate``: blocks are taken until
    ``ceil(num_tokens / block_size)`` are held.
    """
    return (num_tokens + block_size - 1) // block_size


def slot_to_block_offset(slot, block_size):
    """Physical (block, offset-in-block) of a flat slot ``block * block_size + offset``.

    Tokens fill a block in order and spill into the next physical block
    ("vLLM 部署深度指南", section PagedAttention 方案, logical-view figure).
    """
    return slot // block_size, slot % block_size


def logical_to_physical(block_table_row, j, block_size):
    """Physical (block, offset) of logical token ``j`` of one sequence.

    Logical block ``j // block_size`` is looked up in the sequence's block table
    ("vLLM GitHub 项目…", section 二 item 1; "vLLM 部署深度指南", logical-view figure);
    the token sits at offset ``j % block_size`` inside that physical block.
    """
    return int(block_table_row[j // block_size]), j % block_size


def gather_kv(pool, block_table_row, context_len, block_size):
    """Contiguous copies (raw bits) of one sequence's K and V: ``[L, Hkv, D]`` each.

    ``pool`` has shape ``[num_blocks, block_size, 2, Hkv, D]`` (raw bits).
    """
    hkv, d = pool.shape[3], pool.shape[4]
    k = np.empty((context_len, hkv, d), dtype=pool.dtype)
    v = np.empty((context_len, hkv, d), dtype=pool.dtype)
    for j in range(context_len):
        blk, t = logical_to_physical(block_table_row, j, block_size)
        k[j] = pool[blk, t, 0]
        v[j] = pool[blk, t, 1]
    return k, v


# --------------------------------------------------------------------------
# reshape_and_cache: the per-step KV write
# --------------------------------------------------------------------------

def reshape_and_cache(pool, k, v, slot_mapping, src_dtype, kv_dtype, kv_scale=1.0):
    """Return a copy of ``pool`` with each new token's K and V written at its slot.

    ``k``, ``v``: ``[n_tokens, Hkv, D]`` raw bits of ``src_dtype``.
    ``slot_mapping[n] < 0`` marks a padding token and writes nothing.
    For a 16-bit cache the element bits are copied unchanged (``src_dtype`` must
    equal ``kv_dtype``); for an E4M3 cache each element is quantised with
    :func:`fp8_quantise`.  This is the "write to physical block" step of
    ``append_kv`` ("vLLM 部署深度指南", section 代码层面理解), with the slot naming
    the physical block and offset.
    """
    out = pool.copy()
    block_size = pool.shape[1]
    for n, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, t = slot_to_block_offset(int(slot), block_size)
        if kv_dtype == "e4m3":
            out[blk, t, 0] = fp8_quantise(k[n], src_dtype, kv_scale)
            out[blk, t, 1] = fp8_quantise(v[n], src_dtype, kv_scale)
        else:
            if src_dtype != kv_dtype:
                raise ValueError("a 16-bit cache takes sources of its own dtype")
            out[blk, t, 0] = k[n]
            out[blk, t, 1] = v[n]
    return out


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def kv_values(bits, kv_dtype, kv_scale):
    """float64 values of cached K or V elements (dequantised for E4M3)."""
    if kv_dtype == "e4m3":
        return fp8_dequantise(bits, kv_scale)
    return widen(bits, kv_dtype)


def attention_contiguous(q, k, v, scale):
    """Single-query attention of every query head over contiguous K/V, float64.

    ``q``: ``[Hq, D]``; ``k``, ``v``: ``[L, Hkv, D]`` (float64 values).
    Query head ``h`` reads KV head ``h // G`` with ``G = Hq / Hkv`` (query heads
    that share a KV head are consecutive).  Per head:
    ``softmax(scale * q_h . K^T) . V``.  ``L = 0`` gives zeros.
    """
    hq, d = q.shape
    L, hkv = k.shape[0], k.shape[1]
    assert hq % hkv == 0
    g = hq // hkv
    out = np.zeros((hq, d), dtype=np.float64)
    if L == 0:
        return out
    for h in range(hq):
        kh = k[:, h // g, :]                 # [L, D]
        vh = v[:, h // g, :]
        s = scale * (kh @ q[h])              # [L]
        p = np.exp(s - s.max())
        p = p / p.sum()
        out[h] = p @ vh
    return out


def paged_decode(q_bits, q_dtype, pool, block_tables, context_lens, scale,
                 kv_dtype, kv_scale=1.0):
    """Paged decode: gather each sequence through its block table, then attend.

    ``q_bits``: ``[B, Hq, D]`` raw bits; ``pool``: ``[NB, BS, 2, Hkv, D]`` raw bits;
    ``block_tables``: ``[B, max_blocks]`` int; ``context_lens``: ``[B]`` int.
    Returns float64 ``[B, Hq, D]``.  The result equals standard attention on
    the gathered K/V: paging changes only where K/V live ("vLLM GitHub 项目…",
    section 二; "vLLM 部署深度指南", section PagedAttention 方案).
    """
    block_size = pool.shape[1]
    q = widen(q_bits, q_dtype)
    out = np.zeros(q.shape, dtype=np.float64)
    for i in range(q.shape[0]):
        kb, vb = gather_kv(pool, block_tables[i], int(context_lens[i]), block_size)
        k = kv_values(kb, kv_dtype, kv_scale)
        v = kv_values(vb, kv_dtype, kv_scale)
        out[i] = attention_contiguous(q[i], k, v, scale)
    return out


# --------------------------------------------------------------------------
# Prefill / chunked prefill over the paged cache
# --------------------------------------------------------------------------

def paged_prefill(q_bits, q_dtype, pool, block_tables, context_lens, query_start_loc, scale,
                  kv_dtype, kv_scale=1.0):
    """Causal multi-query attention over the paged cache (a prefill step).

    The pages schedule prefills beside decodes ("vLLM 部署深度指南", section
    Continuous Batching, the scheduler sketch: a waiting sequence's prompt
    tokens join the batch in one step) but do not spell out the attention; the
    plainest reading is causal self-attention: a token at position ``p`` of a
    sequence attends to that sequence's tokens ``0..p``.  For a chunk of the
    prompt the chunk's ``n_i`` tokens are the last ``n_i`` of the ``L_i`` cached
    ones (their K/V are written to the pool first, as for a decode step).

    ``q_bits``: ``[T, Hq, D]`` raw bits, sequence ``i``'s queries in rows
    ``query_start_loc[i] .. query_start_loc[i+1]-1`` at positions
    ``L_i - n_i .. L_i - 1``.  Returns float64 ``[T, Hq, D]``.
    """
    block_size = pool.shape[1]
    q = widen(q_bits, q_dtype)
    out = np.zeros(q.shape, dtype=np.float64)
    for i in range(len(context_lens)):
        L = int(context_lens[i])
        r0, r1 = int(query_start_loc[i]), int(query_start_loc[i + 1])
        n = r1 - r0
        assert 0 <= n <= L, "a sequence's query tokens are among its cached tokens"
        if n == 0:
            continue
        kb, vb = gather_kv(pool, block_tables[i], L, block_size)
        k = kv_values(kb, kv_dtype, kv_scale)
        v = kv_values(vb, kv_dtype, kv_scale)
        for t in range(n):
            pos = L - n + t
            out[r0 + t] = attention_contiguous(q[r0 + t], k[:pos + 1], v[:pos + 1], scale)
    return out


# --------------------------------------------------------------------------
# Split-KV: partial attention over a token range and the log-sum-exp merge
# --------------------------------------------------------------------------

def partial_attention(q, k, v, scale):
    """Un-normalised attention state over one KV partition, float64.

    ``q``: ``[D]``; ``k``, ``v``: ``[n, D]``.  Returns ``(m, l, o)`` with
    ``m = max_j s_j``, ``l = sum_j exp(s_j - m)``, ``o = sum_j exp(s_j - m) v_j``.
    An empty partition returns ``(-inf, 0, 0)``.
    """
    if k.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(v.shape[1], dtype=np.float64)
    s = scale * (k @ q)
    m = s.max()
    w = np.exp(s - m)
    return m, w.sum(), w @ v


def merge_partials(parts):
    """Log-sum-exp merge of partial states ``[(m_p, l_p, o_p), ...]``.

    ``M = max m_p``; each partition is weighted by ``exp(m_p - M)``;
    ``out = sum_p exp(m_p - M) o_p / sum_p exp(m_p - M) l_p``.  Empty partitions
    (``m = -inf``, ``l = 0``) carry zero weight.  All-empty gives zeros.
    """
    ms = np.array([p[0] for p in parts], dtype=np.float64)
    live = np.isfinite(ms)
    d = parts[0][2].shape[0]
    if not live.any():
        return np.zeros(d, dtype=np.float64)
    M = ms[live].max()
    num = np.zeros(d, dtype=np.float64)
    den = 0.0
    for (m, l, o), ok in zip(parts, live):
        if not ok:
            continue
        w = np.exp(m - M)
        num += w * o
        den += w * l
    return num / den


def split_kv_attention(q, k, v, scale, partition_size):
    """Attention computed as partitions of ``partition_size`` tokens plus a merge."""
    L = k.shape[0]
    parts = [partial_attention(q, k[s:s + partition_size], v[s:s + partition_size], scale)
             for s in range(0, max(L, 1), partition_size)]
    return merge_partials(parts)
