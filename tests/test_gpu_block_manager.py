"""The block manager driving the GPU path (GB300).

pa_copy_blocks is checked byte for byte; then a parallel-sampling run -- a
prompt forked into several samples that decode token by token -- is driven
entirely by the native manager (slots, copy-on-write pairs, block tables)
and compared, step by step, with the oracle's manager driving the oracle's
pool and decode.
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as ref
from oracle.block_manager import BlockManager as RefManager
from paged_kv_cache_296_gb300 import binding as pa

from harness import ATOL, bits_of

pytestmark = pytest.mark.gpu


def test_copy_blocks_bit_exact():
    g = torch.Generator().manual_seed(3)
    pool = torch.randint(0, 256, (64, 16, 2, 4, 128), dtype=torch.uint8, generator=g)
    src = torch.randperm(64, generator=g)[:20]
    dst = torch.randperm(64, generator=g)
    dst = dst[~torch.isin(dst, src)][:20]
    pairs = torch.stack([src, dst], 1).to(torch.int64)
    dev = pool.cuda()
    pa.pa_copy_blocks(dev, pairs.cuda())
    want = pool.clone()
    want[dst] = pool[src]
    assert torch.equal(dev.cpu(), want)


def test_copy_blocks_skips_bad_pairs_and_reports():
    pool = torch.arange(8 * 16 * 2 * 2 * 64, dtype=torch.int32).view(torch.float16)
    pool = pool.view(8, 16, 2, 2, 128).cuda()
    before = pool.clone()
    pairs = torch.tensor([[1, 2], [3, 99], [-1, 4]], dtype=torch.int64).cuda()
    pa.pa_device_status(clear=True)
    pa.pa_copy_blocks(pool, pairs)
    assert pa.pa_device_status(clear=True) & 4
    want = before.clone()
    want[2] = before[1]
    assert torch.equal(pool.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("prompt_len,samples", [(37, 4), (32, 3), (5, 2)])
def test_parallel_sampling_driven_by_the_manager(prompt_len, samples):
    hq, hkv, d, nb = 8, 2, 64, 48
    rng = torch.Generator().manual_seed(prompt_len + samples)
    bm = pa.BlockManager(nb)
    rm = RefManager(nb)
    # the pool: N(0,1) everywhere, NaN in every slot no sequence holds yet
    pool = torch.full((nb, 16, 2, hkv, d), float("nan"), dtype=torch.float16)
    opool = bits_of(pool)
    gpool = pool.cuda()
    kc, vc = pa.kv_views(gpool)

    def write(slots, k, v):
        s = torch.tensor(slots, dtype=torch.int64)
        pa.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, s.cuda())
        nonlocal opool
        opool = ref.reshape_and_cache(opool, bits_of(k), bits_of(v), s.numpy(), "f16", "f16")

    def copy(pairs):
        if pairs:
            pa.pa_copy_blocks(gpool, torch.tensor(pairs, dtype=torch.int64).cuda())
            for s_, d_ in pairs:
                opool[d_] = opool[s_]

    bm.allocate(0, prompt_len)
    rm.allocate(0, prompt_len)
    w = 8
    t0, _ = bm.block_tables([0], w)
    assert t0[0].tolist() == rm.block_table(0, w)
    k = torch.randn((prompt_len, hkv, d), generator=rng).half()
    v = torch.randn((prompt_len, hkv, d), generator=rng).half()
    write([rm.tables[0][p // 16] * 16 + p % 16 for p in range(prompt_len)], k, v)
    ids = [0]
    for s in range(1, samples):
        bm.fork(0, s)
        rm.fork(0, s)
        ids.append(s)
    for step in range(20):
        slots, copies = bm.append_batch(ids, [1] * len(ids))
        want_slots, want_copies = [], []
        for s in ids:
            sl, cp = rm.append(s, 1)
            want_slots += sl
            want_copies += cp
        assert slots == want_slots and copies == want_copies
        copy(copies)
        k = torch.randn((len(ids), hkv, d), generator=rng).half()
        v = torch.randn((len(ids), hkv, d), generator=rng).half()
        write(slots, k, v)
        tables, lens = bm.block_tables(ids, w)
        q = torch.randn((len(ids), hq, d), generator=rng).half()
        out = torch.empty_like(q).cuda()
        pa.pa_decode(out, q.cuda(), kc, vc, tables.cuda(), lens.cuda(), 0.125)
        want = ref.paged_decode(bits_of(q), "f16", opool, tables.numpy(), lens.numpy(), 0.125,
                                "f16")
        got = ref.widen(bits_of(out.cpu()), "f16")
        assert np.isfinite(got).all(), f"step {step}: a NaN slot was read"
        assert np.abs(got - want).max() <= ATOL["f16"], f"step {step}"
    # every sample's blocks: the prompt's full blocks shared, the rest private
    full = prompt_len // 16
    for b in rm.tables[0][:full]:
        assert bm.ref_count(b) == samples
    for s in ids:
        bm.free(s)
    assert bm.num_free() == nb


def test_prefix_cached_prefill_equals_the_full_prompt():
    """The pages' system-prompt scenario: a second request with the same 2000
    -token system prompt finds its 125 blocks cached, writes and prefills only
    its own 100 tokens (a chunked prefill over the cached prefix), and its
    outputs equal the oracle's prefill of the whole prompt."""
    hq, hkv, d, nb = 8, 2, 64, 512
    g = torch.Generator().manual_seed(11)
    bm = pa.BlockManager(nb)
    pool = torch.full((nb, 16, 2, hkv, d), float("nan"), dtype=torch.bfloat16).cuda()
    kc, vc = pa.kv_views(pool)
    system = torch.randint(0, 32000, (2000,), generator=g).tolist()
    # K/V of a token stand for the token and its prefix: draw them per request
    # position from the token ids, so equal prefixes give equal K/V
    def kv_for(tokens, start):
        out_k, out_v = [], []
        for p in range(start, len(tokens)):
            gg = torch.Generator().manual_seed(hash((tuple(tokens[:p + 1]),)) & 0x7FFFFFFF)
            out_k.append(torch.randn((hkv, d), generator=gg))
            out_v.append(torch.randn((hkv, d), generator=gg))
        return torch.stack(out_k).bfloat16(), torch.stack(out_v).bfloat16()

    def run(seq_id, tokens):
        cached = bm.allocate_cached(seq_id, tokens)
        n = len(tokens)
        t, lens = bm.block_tables([seq_id], 256)
        slots = [int(t[0, p // 16]) * 16 + p % 16 for p in range(cached, n)]
        k, v = kv_for(tokens, cached)
        pa.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc,
                                torch.tensor(slots, dtype=torch.int64).cuda())
        q = torch.randn((n - cached, hq, d), generator=g).bfloat16()
        out = torch.empty_like(q).cuda()
        qsl = torch.tensor([0, n - cached], dtype=torch.int32)
        pa.pa_prefill(out, q.cuda(), kc, vc, t.cuda(), lens.cuda(), qsl.cuda(), n - cached, 0.125)
        return cached, q, out, t, lens, qsl

    user_a = torch.randint(0, 32000, (100,), generator=g).tolist()
    user_b = torch.randint(0, 32000, (100,), generator=g).tolist()
    c_a, *_ = run(1, system + user_a)
    assert c_a == 0
    c_b, q, out, t, lens, qsl = run(2, system + user_b)
    assert c_b == 2000
    assert bm.ref_count(int(t[0, 0])) == 2
    # the oracle: the whole second prompt's K/V laid out privately, the last
    # 100 tokens as queries
    toks = system + user_b
    k_all, v_all = kv_for(toks, 0)
    nblk = -(-len(toks) // 16)
    opool = np.full((nblk, 16, 2, hkv, d), 0, dtype=np.uint16)
    for p in range(len(toks)):
        opool[p // 16, p % 16, 0] = bits_of(k_all[p])
        opool[p // 16, p % 16, 1] = bits_of(v_all[p])
    want = ref.paged_prefill(bits_of(q), "bf16", opool, np.arange(nblk)[None, :],
                             np.array([len(toks)]), np.array([0, 100]), 0.125, "bf16")
    got = ref.widen(bits_of(out.cpu()), "bf16")
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() <= ATOL["bf16"]
