"""The seeded synthetic inputs follow their recipe (CPU only).

Checks the decode and prefill workloads' shapes and distributions, the block
tables' structure (distinct physical blocks, prefix blocks shared only by a
prompt's own samples, -1 past a sequence's last block), the pool size, the
slots the step writes, the poisoning of every slot the step must not read,
and that a seed fixes every byte.  Lengths and the block permutation are drawn
before anything whose size depends on the heads, so the reduced-head copies
used here have exactly the tables of the full-size workloads.
"""

import dataclasses
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_296_gb300 import workloads as wl

BS = 16

#: (B, Hq, Hkv, D, q dtype, cache dtype) of the five decode workloads.
DECODE_SHAPES = {1: (4, 4, 4, 64, "f16", "f16"), 2: (64, 32, 32, 128, "f16", "f16"),
                 3: (256, 32, 8, 128, "bf16", "bf16"), 4: (128, 32, 8, 128, "f16", "f16"),
                 5: (8, 64, 8, 128, "bf16", "e4m3")}


def test_decode_specs_match_the_recipe():
    for n, shape in DECODE_SHAPES.items():
        s = wl.SPECS[n]
        assert (s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_size, s.q_dtype,
                s.kv_dtype) == shape
        assert s.block_size == BS
    assert wl.SPECS[1].lens == ("fixed", [1, 15, 16, 17]) and wl.SPECS[1].pool == ("fixed", 64)
    assert wl.SPECS[2].lens == ("uniform", 128, 2048)
    assert wl.SPECS[3].lens == ("loguniform", 512, 4096)
    assert wl.SPECS[4].lens == ("shared_prefix", 16, 8, 1024, 256)
    assert wl.SPECS[5].lens == ("uniform", 16384, 32768)
    for n in (2, 3, 4, 5):
        assert wl.SPECS[n].pool == ("factor", 1.25)


def test_prefill_specs_match_the_recipe():
    p1, p2 = wl.PREFILL_SPECS[1], wl.PREFILL_SPECS[2]
    assert (p1.num_seqs, p1.num_q_heads, p1.num_kv_heads, p1.head_size, p1.dtype) == \
        (4, 32, 8, 128, "bf16")
    assert p1.context == ("fixed", [2048] * 4) and p1.query == ("all",)
    assert (p2.num_seqs, p2.num_q_heads, p2.num_kv_heads, p2.head_size, p2.dtype) == \
        (16, 32, 8, 128, "bf16")
    assert p2.context == ("uniform", 2048, 8192) and p2.query == ("chunk", 512)


def _reduced(spec):
    """``spec`` with one KV head of size 8 and the same group size."""
    g = spec.num_q_heads // spec.num_kv_heads
    return dataclasses.replace(spec, num_q_heads=g, num_kv_heads=1, head_size=8)


def _within_sigmas(sample_mean, mean, std, n, k=5.0):
    return abs(sample_mean - mean) <= k * std / math.sqrt(n)


def _nan_rows(pool):
    """[num_blocks, BS] mask: True where a pool slot (K and V of every head) is NaN."""
    x = pool.float() if pool.dtype != torch.float32 else pool
    nan = torch.isnan(x).reshape(x.shape[0], x.shape[1], -1)
    assert torch.equal(nan.all(-1), nan.any(-1)), "a slot is partly poisoned"
    return nan.all(-1).numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_workload_follows_the_recipe(n):
    spec = _reduced(wl.SPECS[n])
    W = wl.make_workload(spec, n, poison=True)        # the seed the bench gives rank 0
    L = W.context_lens.numpy().astype(np.int64)
    T = W.block_tables.numpy().astype(np.int64)
    B = spec.num_seqs
    assert L.shape == (B,) and T.shape[0] == B

    kind = spec.lens[0]
    if kind == "fixed":
        assert L.tolist() == spec.lens[1]
    elif kind == "uniform":
        lo, hi = spec.lens[1:]
        assert L.min() >= lo and L.max() <= hi
        assert _within_sigmas(L.mean(), (lo + hi) / 2, (hi - lo) / math.sqrt(12), B)
    elif kind == "loguniform":
        lo, hi = spec.lens[1:]
        assert L.min() >= lo and L.max() <= hi
        a, b = math.log(lo), math.log(hi)
        assert _within_sigmas(np.log(L).mean(), (a + b) / 2, (b - a) / math.sqrt(12), B)
    else:
        prompts, samples, prefix, suffix_hi = spec.lens[1:]
        assert B == prompts * samples
        assert L.min() >= prefix + 1 and L.max() <= prefix + suffix_hi + 1

    nblk = -(-L // BS)
    for i in range(B):
        assert (T[i, nblk[i]:] == -1).all()
    rows = [T[i, :nblk[i]] for i in range(B)]
    ids = np.concatenate(rows)
    assert ids.min() >= 0 and ids.max() < W.num_blocks
    if kind != "shared_prefix":
        assert len(np.unique(ids)) == len(ids), "two tables name one block"
        needed = int(nblk.sum())
    else:
        pblk = prefix // BS
        pre = []
        for p in range(prompts):
            grp = T[p * samples:(p + 1) * samples, :pblk]
            assert (grp == grp[0]).all(), "a prompt's samples must share its prefix blocks"
            pre.append(grp[0])
        private = np.concatenate([T[i, pblk:nblk[i]] for i in range(B)])
        allids = np.concatenate(pre + [private])
        assert len(np.unique(allids)) == len(allids), "shared only within a prompt"
        needed = prompts * pblk + len(private)
    if spec.pool[0] == "factor":
        assert W.num_blocks == math.ceil(spec.pool[1] * needed)
    else:
        assert W.num_blocks == spec.pool[1]

    # The step writes each sequence's last position, L - 1.
    slots = W.slot_mapping.numpy()
    for i in range(B):
        j = L[i] - 1
        assert slots[i] == T[i, j // BS] * BS + j % BS

    # Poisoning: exactly the cached positions 0..L-2 of every sequence hold numbers.
    live = np.zeros((W.num_blocks, BS), dtype=bool)
    for i in range(B):
        pos = np.arange(L[i] - 1)
        live[T[i, pos // BS], pos % BS] = True
    pool = W.pool_src if spec.kv_dtype == "e4m3" else W.pool
    assert np.array_equal(_nan_rows(pool), ~live)

    # Values: N(0, 1) (q and the new tokens; the pool's live slots).
    for t in (W.q, W.k_new, W.v_new):
        x = t.float().flatten()
        assert _within_sigmas(float(x.mean()), 0.0, 1.0, x.numel())
    x = pool.float().flatten()
    x = x[~torch.isnan(x)]
    assert _within_sigmas(float(x.mean()), 0.0, 1.0, x.numel())
    assert abs(float(x.std()) - 1.0) < 0.05

    if spec.kv_dtype == "e4m3":
        amax = max(float(torch.nan_to_num(W.pool_src, nan=0.0).abs().max()),
                   float(W.k_new.float().abs().max()), float(W.v_new.float().abs().max()))
        assert W.kv_scale == amax / 448.0
    else:
        assert W.kv_scale == 1.0
    assert W.scale == 1.0 / math.sqrt(spec.head_size)


@pytest.mark.parametrize("n", [1, 2])
def test_prefill_workload_follows_the_recipe(n):
    spec = _reduced(wl.PREFILL_SPECS[n])
    W = wl.make_prefill_workload(spec, 10 + n, poison=True)   # the bench's seed on rank 0
    L = W.context_lens.numpy().astype(np.int64)
    T = W.block_tables.numpy().astype(np.int64)
    qsl = W.query_start_loc.numpy().astype(np.int64)
    B = spec.num_seqs
    if spec.context[0] == "fixed":
        assert L.tolist() == spec.context[1]
    else:
        lo, hi = spec.context[1:]
        assert L.min() >= lo and L.max() <= hi
    nq = qsl[1:] - qsl[:-1]
    assert qsl[0] == 0
    if spec.query[0] == "all":
        assert np.array_equal(nq, L)
    else:
        assert np.array_equal(nq, np.minimum(L, spec.query[1]))
    assert W.q.shape[0] == qsl[-1] == W.k_new.shape[0] == W.slot_mapping.shape[0]

    nblk = -(-L // BS)
    ids = np.concatenate([T[i, :nblk[i]] for i in range(B)])
    assert len(np.unique(ids)) == len(ids)
    assert ids.min() >= 0 and ids.max() < W.num_blocks
    assert W.num_blocks == math.ceil(spec.pool[1] * int(nblk.sum()))

    # The queries are each sequence's last n positions, written at their slots;
    # only the positions before them hold numbers.
    slots = W.slot_mapping.numpy()
    live = np.zeros((W.num_blocks, BS), dtype=bool)
    for i in range(B):
        pos = np.arange(L[i] - nq[i], L[i])
        assert np.array_equal(slots[qsl[i]:qsl[i + 1]], T[i, pos // BS] * BS + pos % BS)
        old = np.arange(L[i] - nq[i])
        live[T[i, old // BS], old % BS] = True
    assert np.array_equal(_nan_rows(W.pool), ~live)


def test_a_seed_fixes_every_byte():
    spec = _reduced(wl.SPECS[4])
    a, b = wl.make_workload(spec, 4), wl.make_workload(spec, 4)
    for name in ("context_lens", "block_tables", "pool", "q", "k_new", "v_new", "slot_mapping"):
        assert torch.equal(getattr(a, name).view(torch.uint8) if getattr(a, name).dtype.is_floating_point
                           else getattr(a, name),
                           getattr(b, name).view(torch.uint8) if getattr(b, name).dtype.is_floating_point
                           else getattr(b, name)), name
    c = wl.make_workload(spec, 5)
    assert not torch.equal(a.context_lens, c.context_lens)


def test_reduced_heads_keep_the_full_size_tables():
    full = wl.make_workload(wl.SPECS[1], 1)
    small = wl.make_workload(_reduced(wl.SPECS[1]), 1)
    assert torch.equal(full.context_lens, small.context_lens)
    assert torch.equal(full.block_tables, small.block_tables)
    assert torch.equal(full.slot_mapping, small.slot_mapping)
