"""Pins for the oracle's paged decode, gather, write and split-KV merge (CPU only).

Each test checks the oracle against something other than itself: PyTorch's
scaled_dot_product_attention in float64 (a library routine), invariants the
pages fix (block-id permutation, shared prefix blocks), closed forms
(all-equal keys, a single token, no tokens), brute force in pure Python, and
the pages' block-table figure (tests/golden/block_table_figure.txt).
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import paged_attention as ref

GOLDEN_FIG = os.path.join(os.path.dirname(__file__), "golden", "block_table_figure.txt")


# ---------------------------------------------------------------- helpers

def _f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _scatter_to_pool(ks, vs, num_blocks, block_size, rng):
    """Lay contiguous per-sequence K/V out in a pool through shuffled blocks.

    Test-side construction: sequence i's token j goes to the block the table
    names at position j // block_size, offset j % block_size.  Returns
    (pool, tables).
    """
    hkv, d = ks[0].shape[1], ks[0].shape[2]
    pool = np.full((num_blocks, block_size, 2, hkv, d), _f16_bits(np.nan), dtype=np.uint16)
    perm = rng.permutation(num_blocks)
    nb = [max(1, -(-k.shape[0] // block_size)) for k in ks]
    tables = np.full((len(ks), max(nb)), -1, dtype=np.int64)
    nxt = 0
    for i, (k, v) in enumerate(zip(ks, vs)):
        tables[i, :nb[i]] = perm[nxt:nxt + nb[i]]
        nxt += nb[i]
        for j in range(k.shape[0]):
            b = tables[i, j // block_size]
            pool[b, j % block_size, 0] = k[j]
            pool[b, j % block_size, 1] = v[j]
    return pool, tables


def _random_case(rng, B=3, hq=8, hkv=2, d=16, max_len=45, block_size=16):
    lens = [int(x) for x in rng.integers(1, max_len, B)]
    q = _f16_bits(rng.standard_normal((B, hq, d)))
    ks = [_f16_bits(rng.standard_normal((L, hkv, d))) for L in lens]
    vs = [_f16_bits(rng.standard_normal((L, hkv, d))) for L in lens]
    nb = sum(-(-L // block_size) for L in lens) + 5
    pool, tables = _scatter_to_pool(ks, vs, nb, block_size, rng)
    return q, ks, vs, pool, tables, np.array(lens)


# ---------------------------------------------------------------- library pin

@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1), (6, 3)])
def test_paged_equals_sdpa_on_contiguous(hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    q, ks, vs, pool, tables, lens = _random_case(rng, hq=hq, hkv=hkv)
    scale = 1.0 / math.sqrt(16)
    got = ref.paged_decode(q, "f16", pool, tables, lens, scale, "f16")
    for i in range(len(lens)):
        qt = torch.from_numpy(ref.widen(q[i], "f16"))[None, :, None, :]           # [1,Hq,1,D]
        kt = torch.from_numpy(ref.widen(ks[i], "f16")).permute(1, 0, 2)[None]     # [1,Hkv,L,D]
        vt = torch.from_numpy(ref.widen(vs[i], "f16")).permute(1, 0, 2)[None]
        want = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, scale=scale, enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[i], want, rtol=0, atol=1e-12)


def test_gqa_grouping_is_consecutive_heads():
    # With distinct KV heads, query head h must read KV head h // G; reading
    # h % G instead changes the result (guards against the transposed mapping).
    rng = np.random.default_rng(7)
    q, ks, vs, pool, tables, lens = _random_case(rng, hq=4, hkv=2)
    got = ref.paged_decode(q, "f16", pool, tables, lens, 0.25, "f16")
    i = 0
    k = ref.widen(ks[i], "f16")
    v = ref.widen(vs[i], "f16")
    qq = ref.widen(q[i], "f16")
    for h in range(4):
        s = 0.25 * (k[:, h // 2] @ qq[h])
        p = np.exp(s - s.max()); p /= p.sum()
        np.testing.assert_allclose(got[i, h], p @ v[:, h // 2], atol=1e-13, rtol=0)
    s = 0.25 * (k[:, 1 % 2] @ qq[1])  # the wrong mapping for head 1 (h % G = 1 -> 1, h // G = 0)
    p = np.exp(s - s.max()); p /= p.sum()
    assert np.abs(got[i, 1] - p @ v[:, 1]).max() > 1e-3


# ---------------------------------------------------------------- invariants

def test_block_permutation_invariance_exact():
    rng = np.random.default_rng(3)
    q, ks, vs, pool, tables, lens = _random_case(rng)
    a = ref.paged_decode(q, "f16", pool, tables, lens, 0.3, "f16")
    pi = rng.permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[pi] = pool
    tables2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1)
    b = ref.paged_decode(q, "f16", pool2, tables2, lens, 0.3, "f16")
    assert np.array_equal(a, b)


def test_shared_prefix_equals_private_copies_exact():
    rng = np.random.default_rng(4)
    bs, hkv, d, hq = 16, 2, 16, 4
    prefix_blocks, samples = 3, 4
    nb = prefix_blocks + samples * 2 + prefix_blocks * samples + 4
    pool = _f16_bits(rng.standard_normal((nb, bs, 2, hkv, d)))
    perm = rng.permutation(nb)
    pre = perm[:prefix_blocks]
    priv = perm[prefix_blocks:prefix_blocks + 2 * samples].reshape(samples, 2)
    copies = perm[prefix_blocks + 2 * samples:prefix_blocks + 2 * samples + prefix_blocks * samples]
    copies = copies.reshape(samples, prefix_blocks)
    for s in range(samples):
        pool[copies[s]] = pool[pre]
    shared = np.concatenate([np.tile(pre, (samples, 1)), priv], axis=1)
    private = np.concatenate([copies, priv], axis=1)
    lens = prefix_blocks * bs + rng.integers(1, 2 * bs + 1, samples)
    q = _f16_bits(rng.standard_normal((samples, hq, d)))
    a = ref.paged_decode(q, "f16", pool, shared, lens, 0.25, "f16")
    b = ref.paged_decode(q, "f16", pool, private, lens, 0.25, "f16")
    assert np.array_equal(a, b)


def test_all_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(5)
    L, hkv, d = 37, 2, 16
    k = np.tile(_f16_bits(rng.standard_normal((1, hkv, d))), (L, 1, 1))
    v = _f16_bits(rng.standard_normal((L, hkv, d)))
    pool, tables = _scatter_to_pool([k], [v], 6, 16, rng)
    q = _f16_bits(rng.standard_normal((1, 4, d)))
    got = ref.paged_decode(q, "f16", pool, tables, np.array([L]), 0.7, "f16")
    want = ref.widen(v, "f16").mean(axis=0)      # [Hkv, D]
    for h in range(4):
        np.testing.assert_allclose(got[0, h], want[h // 2], rtol=0, atol=1e-15)


def test_single_token_returns_v0_exactly():
    rng = np.random.default_rng(6)
    k = _f16_bits(rng.standard_normal((1, 2, 16)) * 30)
    v = _f16_bits(rng.standard_normal((1, 2, 16)))
    pool, tables = _scatter_to_pool([k], [v], 3, 16, rng)
    q = _f16_bits(rng.standard_normal((1, 2, 16)))
    got = ref.paged_decode(q, "f16", pool, tables, np.array([1]), 1.0, "f16")
    assert np.array_equal(got[0], ref.widen(v[0], "f16"))


def test_empty_context_gives_zeros():
    pool = np.zeros((2, 16, 2, 1, 8), dtype=np.uint16)
    q = _f16_bits(np.ones((1, 1, 8)))
    got = ref.paged_decode(q, "f16", pool, np.array([[0]]), np.array([0]), 1.0, "f16")
    assert np.array_equal(got, np.zeros((1, 1, 8)))


def test_poisoned_unused_slots_are_never_read():
    # _scatter_to_pool leaves every unused slot NaN: a finite result proves
    # the gather stays inside each sequence's L tokens.
    rng = np.random.default_rng(8)
    q, ks, vs, pool, tables, lens = _random_case(rng)
    assert np.isnan(ref.widen(pool, "f16")).any()
    got = ref.paged_decode(q, "f16", pool, tables, lens, 0.3, "f16")
    assert np.isfinite(got).all()


# ---------------------------------------------------------------- brute force

def _brute(q, ks, vs, lens, scale, hq, hkv):
    """Triple loops in plain Python floats."""
    g = hq // hkv
    out = []
    for i, L in enumerate(lens):
        per_head = []
        for h in range(hq):
            s = []
            for j in range(L):
                s.append(scale * sum(float(q[i][h][dd]) * float(ks[i][j][h // g][dd])
                                     for dd in range(len(q[i][h]))))
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            per_head.append([sum(e[j] / tot * float(vs[i][j][h // g][dd]) for j in range(L))
                             for dd in range(len(q[i][h]))])
        out.append(per_head)
    return np.array(out)


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    hq, hkv, d = [(2, 1, 4), (4, 2, 4), (3, 3, 4), (2, 2, 8)][seed]
    q, ks, vs, pool, tables, lens = _random_case(rng, B=3, hq=hq, hkv=hkv, d=d, max_len=40)
    scale = 0.5
    got = ref.paged_decode(q, "f16", pool, tables, lens, scale, "f16")
    want = _brute(ref.widen(q, "f16").tolist(), [ref.widen(k, "f16").tolist() for k in ks],
                  [ref.widen(v, "f16").tolist() for v in vs], lens, scale, hq, hkv)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_brute_force_tiny_config_shape():
    # The tiny workload's own shape: contexts {1, 15, 16, 17}, 4/4 heads, d 64.
    rng = np.random.default_rng(11)
    lens = [1, 15, 16, 17]
    q = _f16_bits(rng.standard_normal((4, 4, 64)))
    ks = [_f16_bits(rng.standard_normal((L, 4, 64))) for L in lens]
    vs = [_f16_bits(rng.standard_normal((L, 4, 64))) for L in lens]
    pool, tables = _scatter_to_pool(ks, vs, 64, 16, rng)
    got = ref.paged_decode(q, "f16", pool, tables, np.array(lens), 1 / 8, "f16")
    want = _brute(ref.widen(q, "f16").tolist(), [ref.widen(k, "f16").tolist() for k in ks],
                  [ref.widen(v, "f16").tolist() for v in vs], lens, 1 / 8, 4, 4)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- split-KV merge

@pytest.mark.parametrize("part", [1, 5, 16, 64, 512])
def test_split_kv_merge_equals_single_pass(part):
    rng = np.random.default_rng(part)
    L, d = 300, 32
    q = rng.standard_normal(d)
    k = rng.standard_normal((L, d)) * 2
    v = rng.standard_normal((L, d))
    one = ref.partial_attention(q, k, v, 0.4)
    want = one[2] / one[1]
    got = ref.split_kv_attention(q, k, v, 0.4, part)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # and against the library routine
    lib = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None, None], torch.from_numpy(k)[None, None],
        torch.from_numpy(v)[None, None], scale=0.4)[0, 0, 0].numpy()
    np.testing.assert_allclose(got, lib, rtol=0, atol=1e-12)


def test_merge_ignores_empty_partitions():
    rng = np.random.default_rng(9)
    q, k, v = rng.standard_normal(8), rng.standard_normal((20, 8)), rng.standard_normal((20, 8))
    full = ref.partial_attention(q, k, v, 1.0)
    empty = ref.partial_attention(q, k[:0], v[:0], 1.0)
    got = ref.merge_partials([empty, full, empty])
    np.testing.assert_allclose(got, full[2] / full[1], rtol=0, atol=1e-15)
    assert np.array_equal(ref.merge_partials([empty]), np.zeros(8))


def test_merge_is_exact_log_sum_exp_for_far_apart_maxima():
    # Partitions whose maxima differ by hundreds: the merge must not overflow.
    q = np.array([1.0])
    k = np.array([[0.0], [500.0], [-400.0]])
    v = np.array([[1.0], [2.0], [3.0]])
    got = ref.split_kv_attention(q, k, v, 1.0, 1)
    assert got[0] == 2.0


# ---------------------------------------------------------------- figure and write

def _read_figure():
    rows, meta = [], {}
    with open(GOLDEN_FIG, encoding="utf-8") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0].isdigit():
                rows.append(tuple(int(x) for x in parts))
            else:
                meta[parts[0]] = parts[1:]
    return rows, meta


def test_block_table_figure_mapping():
    rows, meta = _read_figure()
    bs = int(meta["block_size"][0])
    table = np.array([int(x) for x in meta["block_table"]])
    tokens = meta["tokens"]
    assert ref.blocks_needed(len(tokens), bs) == int(meta["blocks_needed"][0])
    for j, lb, off, pb in rows:
        assert ref.logical_to_physical(table, j, bs) == (pb, off)
        assert j // bs == lb
    # Write the tokens at (physical block, offset) slots, read them back through the table.
    pool = np.full((3, bs, 2, 1, 1), 0xFFFF, dtype=np.uint16)
    ids = np.arange(len(tokens), dtype=np.uint16).reshape(-1, 1, 1)
    slots = np.array([pb * bs + off for (_, _, off, pb) in rows])
    pool = ref.reshape_and_cache(pool, ids, ids + 100, slots, "f16", "f16")
    k, v = ref.gather_kv(pool, table, len(tokens), bs)
    assert k.ravel().tolist() == list(range(len(tokens)))
    assert v.ravel().tolist() == [100 + j for j in range(len(tokens))]
    assert pool[2, 3, 0, 0, 0] == 0xFFFF          # the figure's empty slot stays untouched


def test_reshape_and_cache_skips_padding_and_copies_bits():
    rng = np.random.default_rng(10)
    pool = np.zeros((4, 16, 2, 2, 8), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, (3, 2, 8)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, (3, 2, 8)).astype(np.uint16)
    out = ref.reshape_and_cache(pool, k, v, np.array([17, -1, 63]), "bf16", "bf16")
    assert np.array_equal(out[1, 1, 0], k[0]) and np.array_equal(out[1, 1, 1], v[0])
    assert np.array_equal(out[3, 15, 0], k[2]) and np.array_equal(out[3, 15, 1], v[2])
    touched = np.zeros((4, 16), bool); touched[1, 1] = touched[3, 15] = True
    assert not out[~touched].any()


def test_reshape_and_cache_fp8_quantises_each_element():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 1, 8)).astype(np.float32)
    kb = x.view(np.uint32)
    pool = np.zeros((1, 16, 2, 1, 8), dtype=np.uint8)
    out = ref.reshape_and_cache(pool, kb, kb, np.array([0, 5]), "f32", "e4m3", 0.01)
    lib = (torch.from_numpy(x) / torch.tensor(0.01, dtype=torch.float32)).clamp(-448, 448)
    lib = lib.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(out[0, 0, 0], lib[0]) and np.array_equal(out[0, 5, 1], lib[1])


def test_fp8_decode_uses_dequantised_cache():
    rng = np.random.default_rng(13)
    L, hkv, d = 20, 1, 8
    src = rng.standard_normal((L, hkv, d)).astype(np.float32)
    scale = float(np.abs(src).max() / 448.0)
    codes = ref.fp8_quantise(src.view(np.uint32), "f32", scale)
    pool = np.zeros((2, 16, 2, hkv, d), dtype=np.uint8)
    for j in range(L):
        pool[j // 16, j % 16, 0] = codes[j]
        pool[j // 16, j % 16, 1] = codes[j]
    q = _f16_bits(rng.standard_normal((1, 2, d)))
    got = ref.paged_decode(q, "f16", pool, np.array([[0, 1]]), np.array([L]), 0.3, "e4m3", scale)
    kv = ref.fp8_dequantise(codes, scale)
    want = ref.attention_contiguous(ref.widen(q[0], "f16"), kv, kv, 0.3)
    np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- small helpers

def test_slot_to_block_offset_fills_each_block_in_order():
    # Walking the flat slots in order with a counter (no division) must fill
    # offsets 0..BS-1 of block 0, then of block 1, and so on: the pages'
    # tokens-fill-a-block-then-spill rule.
    for bs in (4, 16):
        blk, off = 0, 0
        for slot in range(7 * bs + 3):
            assert ref.slot_to_block_offset(slot, bs) == (blk, off)
            off += 1
            if off == bs:
                blk, off = blk + 1, 0


def test_kv_values_match_torch_casts():
    # 16-bit caches: every bit pattern widens exactly as PyTorch widens it.
    bits = np.arange(1 << 16, dtype=np.uint16)
    for name, dt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        want = torch.from_numpy(bits.view(np.int16).copy()).view(dt).to(torch.float64).numpy()
        with np.errstate(invalid="ignore"):   # the NaN patterns
            got = ref.kv_values(bits, name, 1.0)
        same = (got == want) | (np.isnan(got) & np.isnan(want))
        assert same.all(), name
    # E4M3 cache: every code decoded by PyTorch's float8_e4m3fn, times float32(kv_scale).
    codes = np.arange(256, dtype=np.uint8)
    kv_scale = 0.0371
    dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    want = dec * np.float64(np.float32(kv_scale))
    got = ref.kv_values(codes, "e4m3", kv_scale)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.isnan(got[~finite]).all()


def test_narrow_f32_rounds_like_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-40, 39, 100000),
                        # exact ties between neighbouring float32 values, both ways
                        (np.float64(1.0) + np.arange(1, 1001) * 2.0 ** -23) + 2.0 ** -24,
                        [0.0, -0.0, np.inf, -np.inf, 3.5e38, 1e-46, -1e-46]])
    want = torch.from_numpy(x).to(torch.float32).numpy()
    with np.errstate(over="ignore"):          # 3.5e38 rounds to inf
        got = ref.narrow_f32(x)
    assert got.dtype == np.float32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
