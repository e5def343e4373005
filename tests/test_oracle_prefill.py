"""Pins for the oracle's causal paged prefill (CPU only).

``ref.paged_prefill`` is checked against things other than itself: PyTorch's
scaled_dot_product_attention with an explicit offset-causal mask (a library
routine), the decode oracle (a prefill chunk of one token per sequence is a
decode step), brute force with explicit loops on tiny shapes, and the closed
forms of special cases (the first prompt token returns v0; all-equal keys give
the running mean of V; the block layout does not matter).
"""

import math

import numpy as np
import pytest
import torch

from oracle import paged_attention as ref


def _f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _case(rng, lens, nq, hq=8, hkv=2, d=16, block_size=16, spare=3):
    """Per-sequence K/V of ``lens`` tokens in a shuffled pool, q for the last
    ``nq[i]`` tokens of each sequence.  Returns (q_bits [T,Hq,D], ks, vs, pool,
    tables, qsl)."""
    ks = [_f16_bits(rng.standard_normal((L, hkv, d))) for L in lens]
    vs = [_f16_bits(rng.standard_normal((L, hkv, d))) for L in lens]
    nb = [max(1, -(-L // block_size)) for L in lens]
    nblocks = sum(nb) + spare
    pool = np.full((nblocks, block_size, 2, hkv, d), _f16_bits(np.nan), dtype=np.uint16)
    perm = rng.permutation(nblocks)
    tables = np.full((len(lens), max(nb)), -1, dtype=np.int64)
    nxt = 0
    for i, L in enumerate(lens):
        tables[i, :nb[i]] = perm[nxt:nxt + nb[i]]
        nxt += nb[i]
        for j in range(L):
            b = tables[i, j // block_size]
            pool[b, j % block_size, 0] = ks[i][j]
            pool[b, j % block_size, 1] = vs[i][j]
    qsl = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    q = _f16_bits(rng.standard_normal((int(qsl[-1]), hq, d)))
    return q, ks, vs, pool, tables, qsl


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (6, 3)])
def test_prefill_equals_sdpa_with_offset_causal_mask(hq, hkv):
    rng = np.random.default_rng(hq + 10 * hkv)
    lens, nq = [40, 17, 33, 5], [40, 3, 16, 5]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, nq, hq=hq, hkv=hkv)
    scale = 1.0 / math.sqrt(16)
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, scale, "f16")
    for i, (L, n) in enumerate(zip(lens, nq)):
        qt = torch.from_numpy(ref.widen(q[qsl[i]:qsl[i + 1]], "f16")).permute(1, 0, 2)[None]
        kt = torch.from_numpy(ref.widen(ks[i], "f16")).permute(1, 0, 2)[None]   # [1,Hkv,L,D]
        vt = torch.from_numpy(ref.widen(vs[i], "f16")).permute(1, 0, 2)[None]
        # query t sits at position L - n + t and may see keys 0 .. L - n + t
        allowed = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        want = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=allowed, scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(got[qsl[i]:qsl[i + 1]], want.numpy(), rtol=0, atol=1e-12)


def test_one_query_per_sequence_is_a_decode_step():
    rng = np.random.default_rng(5)
    lens = [1, 16, 29, 64]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, [1, 1, 1, 1])
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.3, "f16")
    want = ref.paged_decode(q, "f16", pool, tables, np.array(lens), 0.3, "f16")
    assert np.array_equal(got, want)


def test_first_prompt_token_returns_v0_and_equal_keys_give_running_mean():
    rng = np.random.default_rng(6)
    lens = [23]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, [23], hq=2, hkv=1)
    # every key equal: each query's output is the mean of V over positions 0..p
    k0 = ks[0][0].copy()
    for j in range(23):
        b = tables[0, j // 16]
        pool[b, j % 16, 0] = k0
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.7, "f16")
    v = ref.widen(vs[0], "f16")                       # [L, 1, D]
    for t in range(23):
        np.testing.assert_allclose(got[t, 0], v[:t + 1, 0].mean(axis=0), atol=1e-12, rtol=0)
    assert np.array_equal(got[0, 1], v[0, 0])          # position 0 sees only itself


def test_block_permutation_invariance_exact():
    rng = np.random.default_rng(8)
    lens, nq = [50, 20], [30, 20]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, nq)
    a = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.25, "f16")
    pi = rng.permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[pi] = pool
    tables2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1)
    b = ref.paged_prefill(q, "f16", pool2, tables2, np.array(lens), qsl, 0.25, "f16")
    assert np.array_equal(a, b)


def test_causality_later_tokens_do_not_change_earlier_outputs():
    # Changing the K/V of the last cached token changes only the last query's output.
    rng = np.random.default_rng(9)
    lens, nq = [37], [12]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, nq)
    a = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.4, "f16")
    b_, t_ = tables[0, 36 // 16], 36 % 16
    pool[b_, t_, 1] = _f16_bits(rng.standard_normal(pool.shape[3:]))
    b = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.4, "f16")
    assert np.array_equal(a[:-1], b[:-1])
    assert not np.array_equal(a[-1], b[-1])


@pytest.mark.parametrize("seed", range(3))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(200 + seed)
    hq, hkv, d = [(2, 1, 4), (4, 2, 4), (3, 3, 8)][seed]
    lens, nq = [9, 4, 18], [9, 2, 5]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, nq, hq=hq, hkv=hkv, d=d)
    scale = 0.6
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, scale, "f16")
    qv = ref.widen(q, "f16").tolist()
    g = hq // hkv
    for i, (L, n) in enumerate(zip(lens, nq)):
        k = ref.widen(ks[i], "f16").tolist()
        v = ref.widen(vs[i], "f16").tolist()
        for t in range(n):
            pos = L - n + t
            for h in range(hq):
                qh = qv[qsl[i] + t][h]
                s = [scale * sum(qh[e] * k[j][h // g][e] for e in range(d)) for j in range(pos + 1)]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                z = sum(w)
                want = [sum(w[j] * v[j][h // g][e] for j in range(pos + 1)) / z for e in range(d)]
                np.testing.assert_allclose(got[qsl[i] + t, h], want, rtol=0, atol=1e-12)


def test_sequences_without_queries_are_skipped():
    rng = np.random.default_rng(10)
    lens, nq = [20, 35, 8], [0, 4, 0]
    q, ks, vs, pool, tables, qsl = _case(rng, lens, nq)
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, 0.3, "f16")
    assert got.shape == (4, 8, 16)
    one = ref.paged_prefill(q, "f16", pool, tables[1:2], np.array(lens[1:2]),
                            np.array([0, 4]), 0.3, "f16")
    assert np.array_equal(got, one)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4)])
def test_e4m3_prefill_equals_sdpa_on_library_dequantised_codes(hq, hkv):
    # The cache holds E4M3 codes; their values are decoded here by PyTorch's
    # float8_e4m3fn type (a library routine, not the oracle's decoder) and
    # scaled by kv_scale, then attended by scaled_dot_product_attention.
    rng = np.random.default_rng(40 + hq)
    # a kv_scale exact in fp32: the cache's scale is an fp32 value on both sides
    lens, nq, d, bs, kv_scale = [40, 17, 33], [40, 3, 16], 16, 16, 0.375
    nb = [-(-L // bs) for L in lens]
    nblocks = sum(nb) + 2
    pool = np.full((nblocks, bs, 2, hkv, d), 0x7F, dtype=np.uint8)  # NaN codes where unused
    perm = rng.permutation(nblocks)
    tables = np.full((len(lens), max(nb)), -1, dtype=np.int64)
    codes = []
    nxt = 0
    for i, L in enumerate(lens):
        # any code but the two NaNs (0x7F, 0xFF)
        c = (rng.integers(0, 0x7F, (L, 2, hkv, d)) | (rng.integers(0, 2, (L, 2, hkv, d)) << 7))
        c = c.astype(np.uint8)
        codes.append(c)
        tables[i, :nb[i]] = perm[nxt:nxt + nb[i]]
        nxt += nb[i]
        for j in range(L):
            pool[tables[i, j // bs], j % bs] = c[j]
    qsl = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    q = _f16_bits(rng.standard_normal((int(qsl[-1]), hq, d)))
    scale = 1.0 / math.sqrt(d)
    got = ref.paged_prefill(q, "f16", pool, tables, np.array(lens), qsl, scale, "e4m3", kv_scale)
    for i, (L, n) in enumerate(zip(lens, nq)):
        vals = torch.from_numpy(codes[i]).view(torch.float8_e4m3fn).to(torch.float64) * kv_scale
        kt = vals[:, 0].permute(1, 0, 2)[None]   # [1, Hkv, L, D]
        vt = vals[:, 1].permute(1, 0, 2)[None]
        qt = torch.from_numpy(ref.widen(q[qsl[i]:qsl[i + 1]], "f16")).permute(1, 0, 2)[None]
        allowed = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        want = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=allowed, scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(got[qsl[i]:qsl[i + 1]], want.numpy(), rtol=0, atol=1e-12)
