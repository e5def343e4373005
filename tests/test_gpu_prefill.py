"""Paged prefill on the GPU against the float64 oracle (GB300).

Each case writes the step's query tokens' K/V into the pool with
pa_reshape_and_cache (bit-exact against the oracle's write), then runs
pa_prefill and compares every output with ``oracle.paged_prefill`` on the
oracle's own pool.  Unused and not-yet-written slots hold NaN, so a stray read
shows up.  Full-size workloads are checked on sampled rows: the query at
position p of a sequence is the last query of that sequence cut to p + 1
tokens, which the oracle computes on its own.
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as ref
from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300 import workloads as wl

import harness as H
from harness import ATOL, ULP1, bits_of
from oracle import e4m3

pytestmark = pytest.mark.gpu


def gpu_prefill(W):
    dev = "cuda"
    pool = W.pool.to(dev, copy=True)
    kc, vc = pa.kv_views(pool)
    if W.q.shape[0]:
        pa.pa_reshape_and_cache(W.k_new.to(dev), W.v_new.to(dev), kc, vc, W.slot_mapping.to(dev))
    out = torch.full(W.q.shape, float("nan"), dtype=W.q.dtype, device=dev)
    pa.pa_prefill(out, W.q.to(dev), kc, vc, W.block_tables.to(dev), W.context_lens.to(dev),
                  W.query_start_loc.to(dev), W.max_query_len, W.scale)
    return out, pool


def oracle_pool(W):
    d = W.spec.dtype
    return ref.reshape_and_cache(bits_of(W.pool.cpu()), bits_of(W.k_new.cpu()),
                                 bits_of(W.v_new.cpu()), W.slot_mapping.cpu().numpy(), d, d)


def check_close(got, want, dtype, what):
    bound = np.maximum(ATOL[dtype],
                       ULP1[dtype] * np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30)))))
    err = np.abs(got - want)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err "
                           f"{np.nanmax(err):.3e} at {np.argwhere(bad)[:3].tolist()}")


def full_check(W):
    out, pool = gpu_prefill(W)
    opool = oracle_pool(W)
    assert np.array_equal(bits_of(pool.cpu()), opool), "pool after the write differs"
    got = ref.widen(bits_of(out.cpu()), W.spec.dtype)
    assert np.isfinite(got).all(), "NaN output: a slot not yet written or unused was read"
    want = ref.paged_prefill(bits_of(W.q.cpu()), W.spec.dtype, opool, W.block_tables.cpu().numpy(),
                             W.context_lens.cpu().numpy(), W.query_start_loc.cpu().numpy(),
                             W.scale, W.spec.dtype)
    check_close(got, want, W.spec.dtype, W.spec.name)


def random_prefill_spec(seed):
    r = np.random.default_rng(seed)
    d = int(r.choice([64, 128]))
    g = int(r.choice([1, 2, 3, 4, 8]))
    hkv = int(r.choice([1, 2, 3]))
    dt = str(r.choice(["f16", "bf16"]))
    B = int(r.integers(1, 5))
    lens = [int(x) for x in r.integers(1, 160, B)]
    kind = r.integers(0, 3)
    if kind == 0:
        nq = lens                                            # whole prompts
    elif kind == 1:
        nq = [int(r.integers(0, L + 1)) for L in lens]       # chunks over cached prefixes
    else:
        nq = [min(L, int(r.choice([1, 15, 16, 17, 64]))) for L in lens]
    return wl.PrefillSpec(f"random prefill {seed}", B, hkv * g, hkv, d, dt, ("fixed", lens),
                          ("fixed", nq), ("factor", 1.5))


@pytest.mark.parametrize("seed", H.seeds(24))
def test_random_shapes(seed):
    W = wl.make_prefill_workload(random_prefill_spec(seed), 3000 + seed, poison=True)
    full_check(W)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("head_size,group", [(128, 1), (128, 4), (64, 8), (128, 6)])
def test_tile_edges(dtype, head_size, group):
    # query counts around the 128-row tile, the 256-row CTA and the 16-token block
    lens = [63, 64, 65, 200, 129, 16, 1]
    nq = [63, 64, 65, 130, 1, 16, 1]
    spec = wl.PrefillSpec("tile edges", len(lens), 2 * group, 2, head_size, dtype,
                          ("fixed", lens), ("fixed", nq), ("factor", 1.3))
    full_check(wl.make_prefill_workload(spec, 71, poison=True))


def test_large_pool_runs_in_bands_with_a_partial_last_band():
    # A pool larger than half of L2 puts the tiles of one (sequence, KV head)
    # in adjacent bands of 8; 700 queries x 4 heads per KV head are 11 tiles
    # of 256 rows, so the last band holds 3.
    spec = wl.PrefillSpec("large pool", 3, 8, 2, 128, "bf16", ("fixed", [900, 1500, 760]),
                          ("fixed", [700, 300, 650]), ("fixed", 4300))
    W = wl.make_prefill_workload(spec, 23, poison=True)
    assert W.pool.numel() * W.pool.element_size() > 64 * 1024 * 1024
    full_check(W)


def test_one_query_per_sequence_matches_decode():
    # A chunk of one token per sequence is a decode step: both kernels agree
    # within the tolerance (they round differently).
    spec = wl.PrefillSpec("decode-shaped", 6, 32, 8, 128, "bf16",
                          ("fixed", [1, 17, 300, 1000, 33, 2048]), ("chunk", 1))
    W = wl.make_prefill_workload(spec, 5)
    out, pool = gpu_prefill(W)
    kc, vc = pa.kv_views(pool)
    dec = torch.empty_like(out)
    pa.pa_decode(dec, W.q.cuda(), kc, vc, W.block_tables.cuda(), W.context_lens.cuda(), W.scale)
    a = out.float().cpu().numpy()
    b = dec.float().cpu().numpy()
    assert np.abs(a - b).max() <= 2 * ATOL["bf16"]


@pytest.mark.parametrize("n", sorted(wl.PREFILL_SPECS))
def test_full_size_sampled_rows(n):
    W = wl.make_prefill_workload(wl.PREFILL_SPECS[n], 10 + n, device="cuda")
    out, pool = gpu_prefill(W)
    dt = W.spec.dtype
    got_all = ref.widen(bits_of(out.cpu()), dt)
    assert np.isfinite(got_all).all()
    lens = W.context_lens.cpu().numpy()
    qsl = W.query_start_loc.cpu().numpy()
    tables = W.block_tables.cpu().numpy()
    rng = np.random.default_rng(n)
    for i in range(W.spec.num_seqs):
        nq = int(qsl[i + 1] - qsl[i])
        L = int(lens[i])
        for t in sorted({0, nq - 1, int(rng.integers(nq)), int(rng.integers(nq))}):
            pos = L - nq + t
            nb = pos // 16 + 1
            blocks = tables[i, :nb].astype(np.int64)
            # the sequence cut to pos + 1 tokens; its one query is the last token
            sub = bits_of(pool[torch.from_numpy(blocks).cuda()].cpu())
            want = ref.paged_prefill(bits_of(W.q[qsl[i] + t:qsl[i] + t + 1].cpu()), dt, sub,
                                     np.arange(nb)[None, :], np.array([pos + 1]),
                                     np.array([0, 1]), W.scale, dt)
            check_close(got_all[qsl[i] + t][None], want, dt, f"seq {i} token {t}")


def test_long_context_chunk_sampled_rows():
    """A 512-query chunk at the end of 65536- and 40000-token contexts (512 and
    313 chunks of 128 keys per tile): sampled rows against the oracle on the
    sequence cut to each row."""
    spec = wl.PrefillSpec("long context chunk", 2, 32, 8, 128, "bf16", ("fixed", [65536, 40000]),
                          ("chunk", 512), ("factor", 1.05))
    W = wl.make_prefill_workload(spec, 31, device="cuda")
    out, pool = gpu_prefill(W)
    assert pa.pa_device_status(clear=True) == 0
    got_all = ref.widen(bits_of(out.cpu()), "bf16")
    assert np.isfinite(got_all).all()
    lens = W.context_lens.cpu().numpy()
    qsl = W.query_start_loc.cpu().numpy()
    tables = W.block_tables.cpu().numpy()
    rng = np.random.default_rng(31)
    for i in range(2):
        nq = int(qsl[i + 1] - qsl[i])
        L = int(lens[i])
        for t in sorted({0, nq - 1, int(rng.integers(nq))}):
            pos = L - nq + t
            nb = pos // 16 + 1
            blocks = tables[i, :nb].astype(np.int64)
            sub = bits_of(pool[torch.from_numpy(blocks).cuda()].cpu())
            want = ref.paged_prefill(bits_of(W.q[qsl[i] + t:qsl[i] + t + 1].cpu()), "bf16", sub,
                                     np.arange(nb)[None, :], np.array([pos + 1]),
                                     np.array([0, 1]), W.scale, "bf16")
            check_close(got_all[qsl[i] + t][None], want, "bf16", f"seq {i} token {t}")


def test_run_to_run_bitwise_deterministic():
    W = wl.make_prefill_workload(wl.PREFILL_SPECS[2], 12, device="cuda")
    first, _ = gpu_prefill(W)
    for _ in range(3):
        again, _ = gpu_prefill(W)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_bad_query_layout_is_reported_and_skipped():
    # Sequence 1 claims more queries than it has tokens: its rows stay untouched,
    # the device status raises bit 2, the other sequences are still right.
    spec = wl.PrefillSpec("bad layout", 3, 8, 2, 64, "f16", ("fixed", [30, 10, 40]),
                          ("fixed", [30, 10, 40]))
    W = wl.make_prefill_workload(spec, 8)
    opool = oracle_pool(W)
    want = ref.paged_prefill(bits_of(W.q), "f16", opool, W.block_tables.numpy(),
                             W.context_lens.numpy(), W.query_start_loc.numpy(), W.scale, "f16")
    W.context_lens[1] = 5                      # now 10 queries > 5 tokens
    pa.pa_device_status(clear=True)
    out, _ = gpu_prefill(W)
    assert pa.pa_device_status(clear=True) & 2
    got = ref.widen(bits_of(out.cpu()), "f16")
    assert np.isnan(got[30:40]).all(), "rows of the rejected sequence were written"
    check_close(got[:30], want[:30], "f16", "seq 0")
    check_close(got[40:], want[40:], "f16", "seq 2")


def test_empty_batch_and_no_queries_are_no_ops():
    spec = wl.PrefillSpec("no queries", 2, 4, 4, 64, "f16", ("fixed", [20, 9]), ("fixed", [0, 0]))
    W = wl.make_prefill_workload(spec, 9)
    out, _ = gpu_prefill(W)
    assert out.numel() == 0


@pytest.mark.parametrize("dtype,head_size", [("f16", 64), ("bf16", 128)])
def test_growing_logits_rescale_the_accumulator(dtype, head_size):
    # K grows with the position and q is all ones, so every row's running
    # maximum keeps rising: the kernel must rescale what it has accumulated
    # many times over (and the oracle sees the same values).
    lens, nq = [300, 150, 97], [300, 20, 1]
    spec = wl.PrefillSpec("growing logits", 3, 4, 2, head_size, dtype, ("fixed", lens),
                          ("fixed", nq), ("factor", 1.2))
    W = wl.make_prefill_workload(spec, 17)
    tables = W.block_tables.numpy()
    qsl = W.query_start_loc.numpy()
    slope = 3.2 / head_size                           # log2-scaled logit grows ~0.6 per position
    for i, L in enumerate(lens):
        for p in range(L):
            val = slope * p
            if p < L - nq[i]:
                W.pool[tables[i, p // 16], p % 16, 0] = val
            else:
                W.k_new[qsl[i] + p - (L - nq[i])] = val
    W.q.fill_(1.0)
    full_check(W)


# ---------------------------------------------------------------- an E4M3 cache

def fp8_check(spec, seed, poison=True):
    """The spec's pool values as the fp32 sources of an E4M3 cache, with the
    per-tensor kv_scale = amax / 448 over them and the step's new K/V.  The GPU
    fills its cache through pa_reshape_and_cache; the oracle quantises the same
    values by its own rule.  Both caches must agree byte for byte, then
    pa_prefill must agree with the oracle on the dequantised cache."""
    W = wl.make_prefill_workload(spec, seed, poison=poison)
    dev = "cuda"
    src = W.pool.float()                                  # NaN in unused slots when poisoned
    amax = float(torch.nan_to_num(src, nan=0.0).abs().max())
    if W.k_new.numel():
        amax = max(amax, float(W.k_new.float().abs().max()), float(W.v_new.float().abs().max()))
    kv_scale = amax / 448.0
    nb, bs, _, hkv, d = src.shape
    pool = torch.zeros((nb, bs, 2, hkv, d), dtype=torch.uint8, device=dev)
    kc, vc = pa.kv_views(pool)
    flat = src.reshape(nb * bs, 2, hkv, d).to(dev)
    slots = torch.arange(nb * bs, dtype=torch.int64, device=dev)
    pa.pa_reshape_and_cache(flat[:, 0].contiguous(), flat[:, 1].contiguous(), kc, vc, slots,
                            kv_scale=kv_scale)
    if W.q.shape[0]:
        pa.pa_reshape_and_cache(W.k_new.to(dev), W.v_new.to(dev), kc, vc, W.slot_mapping.to(dev),
                                kv_scale=kv_scale)
    out = torch.full(W.q.shape, float("nan"), dtype=W.q.dtype, device=dev)
    pa.pa_prefill(out, W.q.to(dev), kc, vc, W.block_tables.to(dev), W.context_lens.to(dev),
                  W.query_start_loc.to(dev), W.max_query_len, W.scale, kv_scale=kv_scale)
    dt = W.spec.dtype
    opool = ref.fp8_quantise(bits_of(src), "f32", kv_scale)
    opool = ref.reshape_and_cache(opool, bits_of(W.k_new), bits_of(W.v_new),
                                  W.slot_mapping.numpy(), dt, "e4m3", kv_scale)
    gpool = bits_of(pool.cpu())
    assert np.array_equal(e4m3.is_nan_code(gpool), e4m3.is_nan_code(opool))
    live = ~e4m3.is_nan_code(opool)
    assert np.array_equal(gpool[live], opool[live]), "E4M3 cache bytes differ from the oracle's"
    got = ref.widen(bits_of(out.cpu()), dt)
    assert np.isfinite(got).all(), "NaN output: a slot not yet written or unused was read"
    want = ref.paged_prefill(bits_of(W.q), dt, opool, W.block_tables.numpy(),
                             W.context_lens.numpy(), W.query_start_loc.numpy(), W.scale,
                             "e4m3", kv_scale)
    bound = np.maximum(ATOL["e4m3"],
                       ULP1[dt] * np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30)))))
    bad = ~(np.abs(got - want) <= bound)
    assert not bad.any(), (f"{spec.name}: {bad.sum()} of {bad.size} outside tolerance, max err "
                           f"{np.nanmax(np.abs(got - want)):.3e} at {np.argwhere(bad)[:3].tolist()}")


@pytest.mark.parametrize("seed", H.seeds(12))
def test_e4m3_cache_random_shapes(seed):
    spec = random_prefill_spec(100 + seed)
    fp8_check(spec, 5000 + seed)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("head_size,group", [(128, 4), (64, 8), (128, 1)])
def test_e4m3_cache_tile_and_chunk_edges(dtype, head_size, group):
    # query counts around the 128-row tile and the 256-row CTA, contexts around
    # the 128-key chunk and the 16-token block (V rows past L must read as zero)
    lens = [127, 128, 129, 300, 16, 1, 257]
    nq = [127, 64, 129, 200, 16, 1, 3]
    spec = wl.PrefillSpec("e4m3 edges", len(lens), 2 * group, 2, head_size, dtype,
                          ("fixed", lens), ("fixed", nq), ("factor", 1.3))
    fp8_check(spec, 77)


def test_e4m3_cache_bad_query_layout_is_reported():
    spec = wl.PrefillSpec("e4m3 bad layout", 2, 8, 2, 128, "bf16", ("fixed", [30, 10]),
                          ("fixed", [30, 10]))
    W = wl.make_prefill_workload(spec, 8)
    pool = torch.zeros(W.pool.shape, dtype=torch.uint8, device="cuda")
    kc, vc = pa.kv_views(pool)
    lens = W.context_lens.clone()
    lens[1] = 5                                    # 10 queries > 5 tokens
    out = torch.full(W.q.shape, float("nan"), dtype=W.q.dtype, device="cuda")
    pa.pa_device_status(clear=True)
    pa.pa_prefill(out, W.q.cuda(), kc, vc, W.block_tables.cuda(), lens.cuda(),
                  W.query_start_loc.cuda(), W.max_query_len, W.scale, kv_scale=0.5)
    assert pa.pa_device_status(clear=True) & 2
    assert torch.isnan(out[30:].float()).all()
    assert torch.isfinite(out[:30].float()).all()


@pytest.mark.parametrize("n", sorted(wl.PREFILL_SPECS))
def test_e4m3_cache_full_size_sampled_rows(n):
    """The prefill workloads over an E4M3 cache, run as bench.py runs them
    (runner.PrefillStep): for sampled query rows, the oracle quantises the
    sequence's source values (the step's own K/V at the query positions) by its
    rule, the GPU cache bytes of those blocks must equal it, and the row's
    output must match the oracle on the sequence cut to that row."""
    from paged_kv_cache_296_gb300.runner import PrefillStep
    W = wl.make_prefill_workload(wl.PREFILL_SPECS[n], 10 + n, device="cuda")
    S = PrefillStep(W, kv_dtype="e4m3")
    S.step()
    assert pa.pa_device_status(clear=True) == 0
    dt = W.spec.dtype
    got_all = ref.widen(bits_of(S.out.cpu()), dt)
    assert np.isfinite(got_all).all()
    lens = W.context_lens.cpu().numpy()
    qsl = W.query_start_loc.cpu().numpy()
    tables = W.block_tables.cpu().numpy()
    k_new, v_new = W.k_new.cpu().float(), W.v_new.cpu().float()
    rng = np.random.default_rng(100 + n)
    for i in rng.choice(W.spec.num_seqs, size=min(4, W.spec.num_seqs), replace=False):
        nq = int(qsl[i + 1] - qsl[i])
        L = int(lens[i])
        t = int(rng.integers(nq))
        pos = L - nq + t
        nb = pos // 16 + 1
        blocks = torch.from_numpy(tables[i, :nb].astype(np.int64))
        src = W.pool[blocks.cuda()].cpu().float()                   # [nb, 16, 2, Hkv, D]
        for p in range(L - nq, pos + 1):                             # the step's own tokens
            src[p // 16, p % 16, 0] = k_new[qsl[i] + p - (L - nq)]
            src[p // 16, p % 16, 1] = v_new[qsl[i] + p - (L - nq)]
        opool = ref.fp8_quantise(bits_of(src), "f32", S.kv_scale)
        gpool = bits_of(S.pool[blocks.cuda()].cpu())
        # slots past pos in the last block are not part of the cut sequence
        keep = np.zeros(opool.shape, dtype=bool)
        keep.reshape(nb * 16, -1)[:pos + 1] = True
        assert np.array_equal(gpool[keep], opool[keep]), f"seq {i}: cache bytes differ"
        want = ref.paged_prefill(bits_of(W.q[qsl[i] + t:qsl[i] + t + 1].cpu()), dt, opool,
                                 np.arange(nb)[None, :], np.array([pos + 1]), np.array([0, 1]),
                                 W.scale, "e4m3", S.kv_scale)
        err = np.abs(got_all[qsl[i] + t] - want[0])
        assert err.max() <= ATOL["e4m3"], f"seq {i} token {t}: max err {err.max():.3e}"


def test_e4m3_cache_long_context_chunk_sampled_rows():
    """The long-context chunk over an E4M3 cache: the widening runs 512 and 313
    chunks per tile; sampled rows and their cache bytes against the oracle."""
    from paged_kv_cache_296_gb300.runner import PrefillStep
    spec = wl.PrefillSpec("long context chunk", 2, 32, 8, 128, "bf16", ("fixed", [65536, 40000]),
                          ("chunk", 512), ("factor", 1.05))
    W = wl.make_prefill_workload(spec, 32, device="cuda")
    S = PrefillStep(W, kv_dtype="e4m3")
    S.step()
    assert pa.pa_device_status(clear=True) == 0
    got_all = ref.widen(bits_of(S.out.cpu()), "bf16")
    assert np.isfinite(got_all).all()
    lens = W.context_lens.cpu().numpy()
    qsl = W.query_start_loc.cpu().numpy()
    tables = W.block_tables.cpu().numpy()
    k_new, v_new = W.k_new.cpu().float(), W.v_new.cpu().float()
    rng = np.random.default_rng(32)
    for i in range(2):
        nq = int(qsl[i + 1] - qsl[i])
        L = int(lens[i])
        for t in sorted({nq - 1, int(rng.integers(nq))}):
            pos = L - nq + t
            nb = pos // 16 + 1
            blocks = torch.from_numpy(tables[i, :nb].astype(np.int64))
            src = W.pool[blocks.cuda()].cpu().float()
            for q in range(L - nq, pos + 1):
                src[q // 16, q % 16, 0] = k_new[qsl[i] + q - (L - nq)]
                src[q // 16, q % 16, 1] = v_new[qsl[i] + q - (L - nq)]
            opool = ref.fp8_quantise(bits_of(src), "f32", S.kv_scale)
            gpool = bits_of(S.pool[blocks.cuda()].cpu())
            keep = np.zeros(opool.shape, dtype=bool)
            keep.reshape(nb * 16, -1)[:pos + 1] = True
            assert np.array_equal(gpool[keep], opool[keep]), f"seq {i}: cache bytes differ"
            want = ref.paged_prefill(bits_of(W.q[qsl[i] + t:qsl[i] + t + 1].cpu()), "bf16", opool,
                                     np.arange(nb)[None, :], np.array([pos + 1]),
                                     np.array([0, 1]), W.scale, "e4m3", S.kv_scale)
            err = np.abs(got_all[qsl[i] + t] - want[0])
            assert err.max() <= ATOL["e4m3"], f"seq {i} token {t}: max err {err.max():.3e}"


def test_context_length_past_the_table_is_cut_to_it():
    # A context length beyond max_blocks_per_seq * 16 is read as the table's
    # capacity: no entry past the row is read, and the outputs equal the
    # oracle's on the cut length (the queries are then the last tokens of it).
    spec = wl.PrefillSpec("past the table", 2, 8, 2, 64, "f16", ("fixed", [40, 64]),
                          ("fixed", [8, 16]))
    W = wl.make_prefill_workload(spec, 31, poison=True)
    width = W.block_tables.shape[1]
    lens = W.context_lens.clone()
    lens[1] = width * 16 + 50                    # past the row's capacity
    cut = W.context_lens.clone()
    cut[1] = width * 16
    dev = "cuda"
    pool = W.pool.to(dev, copy=True)
    kc, vc = pa.kv_views(pool)
    pa.pa_reshape_and_cache(W.k_new.to(dev), W.v_new.to(dev), kc, vc, W.slot_mapping.to(dev))
    out = torch.full(W.q.shape, float("nan"), dtype=W.q.dtype, device=dev)
    pa.pa_prefill(out, W.q.to(dev), kc, vc, W.block_tables.to(dev), lens.to(dev),
                  W.query_start_loc.to(dev), W.max_query_len, W.scale)
    opool = oracle_pool(W)
    got = ref.widen(bits_of(out.cpu()), "f16")
    assert np.isfinite(got).all()
    want = ref.paged_prefill(bits_of(W.q), "f16", opool, W.block_tables.numpy(), cut.numpy(),
                             W.query_start_loc.numpy(), W.scale, "f16")
    check_close(got, want, "f16", "cut length")


def test_e4m3_cache_run_to_run_bitwise_deterministic():
    # the converters hand staging buffers and ring slots between proxies:
    # repeated runs at full size must agree bit for bit
    from paged_kv_cache_296_gb300.runner import PrefillStep
    W = wl.make_prefill_workload(wl.PREFILL_SPECS[2], 12, device="cuda")
    S = PrefillStep(W, kv_dtype="e4m3")
    first = S.step().clone()
    for _ in range(10):
        again = S.step()
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    assert pa.pa_device_status(clear=True) == 0


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_block_permutation_invariance_bitwise(kv):
    # Paging changes only where K/V live: moving every block to another
    # physical id (and rewriting the tables and slots to match) leaves every
    # output bit unchanged.
    spec = wl.PrefillSpec("permuted", 5, 16, 4, 128, "bf16", ("fixed", [300, 129, 1000, 64, 517]),
                          ("fixed", [300, 40, 256, 64, 17]), ("factor", 1.4))
    W = wl.make_prefill_workload(spec, 19)

    def run(pool16, tables, slots):
        from paged_kv_cache_296_gb300.runner import PrefillStep
        W.pool, W.block_tables, W.slot_mapping = pool16, tables, slots
        S = PrefillStep(W, kv_dtype=None if kv == "bf16" else "e4m3")
        return S.step().cpu()

    pool0, tables0, slots0 = W.pool.clone(), W.block_tables.clone(), W.slot_mapping.clone()
    a = run(pool0, tables0, slots0)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(W.num_blocks))  # old id -> new id
    pool1 = torch.empty_like(pool0)
    pool1[perm] = pool0
    tables1 = torch.where(tables0 >= 0, perm[tables0.clamp(min=0).long()].to(torch.int32), tables0)
    slots1 = perm[slots0 // 16] * 16 + slots0 % 16
    b = run(pool1, tables1, slots1)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
