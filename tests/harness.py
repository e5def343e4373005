"""Test harness: run one decode step through the CUDA library and through the oracle.

Both sides start from the same seeded Workload (paged_kv_cache_296_gb300.workloads).
The GPU side calls the C ABI through the Python binding; the oracle side takes
the CPU copies of the inputs, never a value the GPU produced.
"""

import os

import numpy as np
import torch

from oracle import paged_attention as ref
from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300.workloads import BLOCK_SIZE

def seeds(n):
    """The seeds of a random-shape sweep: range(n), or range(PA_RANDOM_SEEDS) when
    that environment variable asks for a longer sweep."""
    return range(max(n, int(os.environ.get("PA_RANDOM_SEEDS", "0"))))


#: Attention tolerances (max abs error against the float64 oracle).
ATOL = {"f16": 2e-3, "bf16": 1e-2, "e4m3": 3e-2}

#: Unit in the last place of the output dtype at magnitude 1 (used to widen the
#: bound for tiny contexts, whose outputs can be large: the output rounding
#: alone is half an ulp of |out|).
ULP1 = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}


def bits_of(t):
    """Raw element bits of a CPU tensor as a NumPy array (uint16 / uint8 / uint32)."""
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def gpu_pool(W, device="cuda"):
    """The pool as the GPU path holds it before the step.

    16-bit caches are the generated values; an E4M3 cache is filled from the
    fp32 source values by pa_reshape_and_cache over every slot of the pool.
    """
    spec = W.spec
    if spec.kv_dtype != "e4m3":
        return W.pool.to(device)
    nb, bs, _, hkv, d = W.pool_src.shape
    pool = torch.zeros((nb, bs, 2, hkv, d), dtype=torch.uint8, device=device)
    kc, vc = pa.kv_views(pool)
    chunk = 1 << 16  # token rows per fill call
    src = W.pool_src.reshape(nb * bs, 2, hkv, d)
    for r0 in range(0, nb * bs, chunk):
        r1 = min(nb * bs, r0 + chunk)
        part = src[r0:r1].to(device)
        slots = torch.arange(r0, r1, dtype=torch.int64, device=device)
        pa.pa_reshape_and_cache(part[:, 0].contiguous(), part[:, 1].contiguous(), kc, vc, slots,
                                kv_scale=W.kv_scale)
    return pool


def gpu_step(W, pool, partition_size=0, workspace=None, write=True):
    """reshape_and_cache of the step's new tokens, then paged decode; returns out (device)."""
    dev = pool.device
    kc, vc = pa.kv_views(pool)
    if write:
        pa.pa_reshape_and_cache(W.k_new.to(dev), W.v_new.to(dev), kc, vc, W.slot_mapping.to(dev),
                                kv_scale=W.kv_scale)
    out = torch.empty(W.q.shape, dtype=W.q.dtype, device=dev)
    pa.pa_decode(out, W.q.to(dev), kc, vc, W.block_tables.to(dev), W.context_lens.to(dev),
                 W.scale, kv_scale=W.kv_scale, partition_size=partition_size,
                 workspace=workspace)
    return out


# ---------------------------------------------------------------- oracle side

def oracle_pool_after_step(W):
    """The oracle's pool (raw bits) after the step's write (16-bit caches only)."""
    spec = W.spec
    assert spec.kv_dtype != "e4m3"
    pool = bits_of(W.pool)
    return ref.reshape_and_cache(pool, bits_of(W.k_new), bits_of(W.v_new),
                                 W.slot_mapping.numpy(), spec.q_dtype, spec.kv_dtype)


def oracle_decode_full(W, pool_bits):
    spec = W.spec
    return ref.paged_decode(bits_of(W.q), spec.q_dtype, pool_bits, W.block_tables.numpy(),
                            W.context_lens.numpy(), W.scale, spec.kv_dtype, W.kv_scale)


def mini_case(W, seq, kv_head):
    """One (sequence, KV head) of a workload as a self-contained small case.

    Returns (blocks, mini) where ``blocks`` are the physical ids the sequence's
    table names and ``mini`` holds the oracle-side arrays: the pool slice of
    those blocks and that head (raw bits, fp32 source for E4M3), a table
    0..n-1, the new token's slot remapped into the slice, and q / k / v of
    that head group.
    """
    spec = W.spec
    L = int(W.context_lens[seq])
    nblk = -(-L // BLOCK_SIZE)
    blocks = W.block_tables[seq, :nblk].numpy().astype(np.int64)
    g = spec.num_q_heads // spec.num_kv_heads
    src = W.pool_src if spec.kv_dtype == "e4m3" else W.pool
    pool_slice = src[torch.from_numpy(blocks)][:, :, :, kv_head:kv_head + 1, :].contiguous()
    slot = int(W.slot_mapping[seq])
    if slot >= 0:
        pos = int(np.nonzero(blocks == slot // BLOCK_SIZE)[0][0])
        slot = pos * BLOCK_SIZE + slot % BLOCK_SIZE
    mini = dict(
        pool=bits_of(pool_slice), table=np.arange(max(nblk, 1))[None, :], L=np.array([L]),
        slot=np.array([slot]),
        q=bits_of(W.q[seq:seq + 1, kv_head * g:(kv_head + 1) * g]),
        k=bits_of(W.k_new[seq:seq + 1, kv_head:kv_head + 1]),
        v=bits_of(W.v_new[seq:seq + 1, kv_head:kv_head + 1]),
    )
    return blocks, mini


def oracle_mini(W, mini):
    """Oracle pool slice after the step and the decode output ``[G, D]`` for a mini case."""
    spec = W.spec
    if spec.kv_dtype == "e4m3":
        pool = ref.fp8_quantise(mini["pool"], "f32", W.kv_scale)
    else:
        pool = mini["pool"]
    pool = ref.reshape_and_cache(pool, mini["k"], mini["v"], mini["slot"], spec.q_dtype,
                                 spec.kv_dtype, W.kv_scale)
    out = ref.paged_decode(mini["q"], spec.q_dtype, pool, mini["table"], mini["L"], W.scale,
                           spec.kv_dtype, W.kv_scale)
    return pool, out[0]


def widen_out(t, dtype):
    return ref.widen(bits_of(t.cpu()), dtype)


def tolerance(spec, ref_out):
    """Per-element bound: the stated tolerance for the cache dtype, widened by
    one output ulp of |ref| where that exceeds it (only large outputs of tiny
    contexts reach that)."""
    atol = ATOL[spec.kv_dtype]
    ulp = ULP1[spec.q_dtype] * np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_out), 1e-30))))
    return np.maximum(atol, ulp)


def assert_close(got, want, spec, what=""):
    bound = tolerance(spec, want)
    err = np.abs(got - want)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outputs outside tolerance; max err "
            f"{np.nanmax(err):.3e}; first at {idx.tolist()} got {got[bad][:5]} want {want[bad][:5]}")
    return float(err.max()) if err.size else 0.0

