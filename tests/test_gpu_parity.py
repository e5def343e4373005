"""GPU parity: the CUDA library against the float64 oracle on the same seeded inputs.

Writes and gathers must match bit for bit; attention must match within the
stated tolerances (fp16 2e-3, bf16 1e-2, fp8-E4M3 cache 3e-2 against the
oracle on the dequantised cache).  Unused pool slots are poisoned with NaN, so
any stray read shows up as a NaN output.  Every call goes through the C ABI.
"""

import numpy as np
import pytest
import torch

from oracle import e4m3
from oracle import paged_attention as ref
from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300 import workloads as wl

import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    pa.load()
    pa.pa_device_status(clear=True)
    yield
    assert pa.pa_device_status(clear=True) == 0, "a kernel raised a device error bit"


# ---------------------------------------------------------------- reshape_and_cache

def _torch_dtype(name):
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


@pytest.mark.parametrize("src,kv", [("f16", "f16"), ("bf16", "bf16"), ("f16", "e4m3"),
                                    ("bf16", "e4m3"), ("f32", "e4m3")])
@pytest.mark.parametrize("head_size", [64, 128])
def test_reshape_and_cache_bit_exact(src, kv, head_size):
    g = torch.Generator().manual_seed(7)
    nb, hkv, n = 40, 3, 200
    if kv == "e4m3":
        pool = torch.randint(0, 256, (nb, 16, 2, hkv, head_size), generator=g, dtype=torch.uint8)
    else:
        pool = torch.randn((nb, 16, 2, hkv, head_size), generator=g).to(_torch_dtype(kv))
    # strided source: each token row padded by 8 elements (a fused-qkv layout)
    stride_pad = 16 if src == "f32" else 8
    full_k = (torch.randn((n, hkv * head_size + stride_pad), generator=g) * 3).to(_torch_dtype(src))
    full_v = (torch.randn((n, hkv * head_size + stride_pad), generator=g) * 3).to(_torch_dtype(src))
    if kv == "e4m3":
        # saturation, NaN, signed zero, tiny values and exact ties on the write path
        specials = torch.tensor([1e4, -1e4, float("nan"), -0.0, 1e-30, float("inf"),
                                 -float("inf"), 0.1]).to(_torch_dtype(src))
        full_k[0, :8] = specials
        full_v[1, :8] = specials
    k = full_k[:, :hkv * head_size].view(n, hkv, head_size)
    v = full_v[:, :hkv * head_size].view(n, hkv, head_size)
    perm = torch.randperm(nb * 16, generator=g)[:n].to(torch.int64)
    perm[::7] = -1                                   # padding tokens
    perm[5] = nb * 16 + 3                            # past the pool: skipped
    kv_scale = 0.037

    dev_pool = pool.cuda()
    kc, vc = pa.kv_views(dev_pool)
    pa.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, perm.cuda(), kv_scale=kv_scale)
    got = H.bits_of(dev_pool.cpu())

    slots = perm.numpy().copy()
    slots[slots >= nb * 16] = -1                     # the oracle's pool has no such slot
    want = ref.reshape_and_cache(H.bits_of(pool), H.bits_of(k.contiguous()),
                                 H.bits_of(v.contiguous()), slots, src, kv, kv_scale)
    if kv == "e4m3":
        nan_w, nan_g = e4m3.is_nan_code(want), e4m3.is_nan_code(got)
        assert np.array_equal(nan_w, nan_g)
        assert np.array_equal(got[~nan_g], want[~nan_w])
        assert nan_w.any()
    else:
        assert np.array_equal(got, want)


# ---------------------------------------------------------------- gather

@pytest.mark.parametrize("kv", ["f16", "bf16", "e4m3"])
def test_gather_bit_exact(kv):
    spec = wl.random_spec(3, head_size=128, group=2, kv_dtype=kv, max_len=90, max_seqs=6)
    W = wl.make_workload(spec, 31, poison=True, table_garbage=True)
    pool = H.gpu_pool(W)
    kc, vc = pa.kv_views(pool)
    lens = W.context_lens.numpy()
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    total = int(cu[-1])
    hkv, d = spec.num_kv_heads, spec.head_size
    ko = torch.zeros((max(total, 1), hkv, d), dtype=pool.dtype, device="cuda")
    vo = torch.zeros_like(ko)
    pa.pa_gather_kv(ko, vo, kc, vc, W.block_tables.cuda(), W.context_lens.cuda(),
                    torch.from_numpy(cu).cuda())
    ko, vo = H.bits_of(ko.cpu()), H.bits_of(vo.cpu())
    if kv == "e4m3":
        opool = ref.fp8_quantise(H.bits_of(W.pool_src), "f32", W.kv_scale)
    else:
        opool = H.bits_of(W.pool)
    for i, L in enumerate(lens):
        k, v = ref.gather_kv(opool, W.block_tables[i].numpy(), int(L), 16)
        for got, want in ((ko[cu[i]:cu[i + 1]], k), (vo[cu[i]:cu[i + 1]], v)):
            if kv == "e4m3":   # NaN codes (poisoned slots) may differ in sign only
                nan = e4m3.is_nan_code(want)
                assert np.array_equal(e4m3.is_nan_code(got), nan)
                assert np.array_equal(got[~nan], want[~nan])
            else:
                assert np.array_equal(got, want)


def _fp32_rounding_boundaries():
    """float32 values a few ulps either side of every E4M3 rounding boundary
    (the midpoints between neighbouring codes, the codes themselves and the
    saturation edge), both signs, plus random float32 bit patterns (NaNs,
    infinities and subnormals among them)."""
    mags = e4m3.decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (mags[:-1] + mags[1:]) / 2
    edges = np.concatenate([mags, mids, [464.0, 480.0]]).astype(np.float32)
    pts = [edges]
    for direction in (np.float32(np.inf), np.float32(-np.inf)):
        x = edges
        for _ in range(3):
            x = np.nextafter(x, direction)
            pts.append(x)
    x = np.concatenate(pts)
    x = np.concatenate([x, -x])
    rnd = np.random.default_rng(5).integers(0, 1 << 32, 1 << 16, dtype=np.uint64)
    return np.concatenate([x, rnd.astype(np.uint32).view(np.float32)])


@pytest.mark.parametrize("src", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("kv_scale", [1.0, 0.037])
def test_fp8_write_exhaustive(src, kv_scale):
    # Every fp16 / bf16 bit pattern (all the write path can see from a 16-bit
    # source), or float32 around every rounding boundary, through
    # pa_reshape_and_cache into an E4M3 cache: byte for byte the oracle's
    # float32 divide then round-to-nearest-even with saturation.  NaN inputs
    # must give a NaN code; its sign is fixed by neither side.
    if src == "f32":
        vals = _fp32_rounding_boundaries()
        x = torch.from_numpy(vals.copy())
    else:
        bits = np.arange(1 << 16, dtype=np.uint16)
        x = torch.from_numpy(bits.view(np.int16).copy()).view(_torch_dtype(src))
    hkv, d = 2, 128
    per_tok = hkv * d
    n = -(-x.numel() // per_tok)
    flat = torch.zeros(n * per_tok, dtype=x.dtype)
    flat[:x.numel()] = x
    k = flat.view(n, hkv, d)
    v = flat.flip(0).contiguous().view(n, hkv, d)
    nb = -(-n // 16)
    g = torch.Generator().manual_seed(11)
    pool = torch.randint(0, 256, (nb, 16, 2, hkv, d), generator=g, dtype=torch.uint8)
    slots = torch.randperm(nb * 16, generator=g)[:n].to(torch.int64)

    dev_pool = pool.cuda()
    kc, vc = pa.kv_views(dev_pool)
    pa.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots.cuda(), kv_scale=kv_scale)
    got = H.bits_of(dev_pool.cpu())
    with np.errstate(over="ignore", invalid="ignore"):
        want = ref.reshape_and_cache(H.bits_of(pool), H.bits_of(k), H.bits_of(v),
                                     slots.numpy(), src, "e4m3", kv_scale)
    nan_w, nan_g = e4m3.is_nan_code(want), e4m3.is_nan_code(got)
    assert np.array_equal(nan_w, nan_g)
    bad = np.flatnonzero(got[~nan_w] != want[~nan_w])
    assert bad.size == 0, f"{bad.size} codes differ, first at {bad[:4]}"


def test_fp8_pool_fill_matches_oracle_encoding():
    spec = wl.random_spec(4, head_size=64, group=4, kv_dtype="e4m3", max_len=60)
    W = wl.make_workload(spec, 41, poison=True)
    got = H.bits_of(H.gpu_pool(W).cpu())
    want = ref.fp8_quantise(H.bits_of(W.pool_src), "f32", W.kv_scale)
    assert np.array_equal(e4m3.is_nan_code(got), e4m3.is_nan_code(want))
    ok = ~e4m3.is_nan_code(want)
    assert np.array_equal(got[ok], want[ok])


# ---------------------------------------------------------------- decode: the five workloads

def _full_check(W, partition_size=0):
    spec = W.spec
    pool = H.gpu_pool(W)
    out = H.gpu_step(W, pool, partition_size=partition_size)
    got = H.widen_out(out, spec.q_dtype)
    assert np.isfinite(got).all(), "NaN/inf output: a poisoned slot was read"
    opool = H.oracle_pool_after_step(W)
    assert np.array_equal(H.bits_of(pool.cpu()), opool), "pool after the write differs"
    want = H.oracle_decode_full(W, opool)
    return H.assert_close(got, want, spec, spec.name)


def test_config1_tiny():
    W = wl.make_workload(wl.SPECS[1], 1, poison=True, table_garbage=True)
    _full_check(W)


@pytest.mark.parametrize("n", [2, 3, 4])
def test_full_size_config_all_outputs(n):
    W = wl.make_workload(wl.SPECS[n], n, poison=True)
    _full_check(W)


def test_config5_long_fp8_sampled():
    """Long-context fp8 workload at full size: every sequence, one KV head each,
    checked against the oracle on the dequantised cache; the pool bytes of
    those heads checked bit for bit."""
    W = wl.make_workload(wl.SPECS[5], 5, poison=True)
    spec = W.spec
    pool = H.gpu_pool(W)
    out = H.gpu_step(W, pool)
    got_all = H.widen_out(out, spec.q_dtype)
    assert np.isfinite(got_all).all()
    g = spec.num_q_heads // spec.num_kv_heads
    rng = np.random.default_rng(5)
    for i in range(spec.num_seqs):
        h = int(rng.integers(spec.num_kv_heads))
        blocks, mini = H.mini_case(W, i, h)
        opool, want = H.oracle_mini(W, mini)
        gpool = H.bits_of(pool[torch.from_numpy(blocks).cuda()][:, :, :, h:h + 1].cpu())
        assert np.array_equal(e4m3.is_nan_code(gpool), e4m3.is_nan_code(opool))
        live = ~e4m3.is_nan_code(opool)
        assert np.array_equal(gpool[live], opool[live])
        H.assert_close(got_all[i, h * g:(h + 1) * g], want, spec, f"seq {i} kv head {h}")


# ---------------------------------------------------------------- decode: sweeps and edges

@pytest.mark.parametrize("seed", H.seeds(24))
def test_random_shapes(seed):
    spec = wl.random_spec(seed)
    W = wl.make_workload(spec, 1000 + seed, poison=True, table_garbage=True)
    if spec.kv_dtype == "e4m3":
        pool = H.gpu_pool(W)
        out = H.gpu_step(W, pool, partition_size=spec.partition_size)
        got = H.widen_out(out, spec.q_dtype)
        for i in range(spec.num_seqs):
            for h in range(spec.num_kv_heads):
                g = spec.num_q_heads // spec.num_kv_heads
                _, mini = H.mini_case(W, i, h)
                _, want = H.oracle_mini(W, mini)
                H.assert_close(got[i, h * g:(h + 1) * g], want, spec, f"{spec.name} s{i} h{h}")
    else:
        _full_check(W, partition_size=spec.partition_size)


EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1000]


@pytest.mark.parametrize("kv,q", [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16"),
                                  ("e4m3", "f16")])
@pytest.mark.parametrize("head_size,group", [(64, 1), (128, 4), (128, 8), (64, 3)])
@pytest.mark.parametrize("part", [16, 48, 0])
def test_edge_context_lengths(kv, q, head_size, group, part):
    spec = wl.Spec("edges", len(EDGE_LENS), 2 * group, 2, head_size, q, kv,
                   ("fixed", EDGE_LENS), ("factor", 1.3))
    W = wl.make_workload(spec, 77, poison=True, table_garbage=True)
    pool = H.gpu_pool(W)
    out = H.gpu_step(W, pool, partition_size=part)
    got = H.widen_out(out, q)
    assert np.isfinite(got).all()
    assert np.array_equal(got[0], np.zeros_like(got[0])), "empty context must give zeros"
    if kv != "e4m3":
        want = H.oracle_decode_full(W, H.oracle_pool_after_step(W))
        H.assert_close(got, want, spec, "edges")
        # context length 1 returns v0 (the token written this step) exactly
        v0 = ref.widen(H.bits_of(W.v_new[1]), kv)
        for h in range(spec.num_q_heads):
            assert np.array_equal(got[1, h], v0[h // group])
    else:
        for i in range(spec.num_seqs):
            for h in range(spec.num_kv_heads):
                _, mini = H.mini_case(W, i, h)
                _, want = H.oracle_mini(W, mini)
                H.assert_close(got[i, h * group:(h + 1) * group], want, spec, f"s{i} h{h}")


def test_all_equal_keys_give_mean_of_v():
    spec = wl.Spec("equal keys", 3, 8, 2, 128, "f16", "f16", ("fixed", [40, 300, 700]))
    W = wl.make_workload(spec, 9)
    # one key row for every token of every sequence
    W.pool[:, :, 0] = W.pool[0, 0, 0]
    W.k_new[:] = W.pool[0, 0, 0]
    out = H.widen_out(H.gpu_step(W, H.gpu_pool(W)), "f16")
    opool = H.oracle_pool_after_step(W)
    for i, L in enumerate(W.context_lens.numpy()):
        _, v = ref.gather_kv(opool, W.block_tables[i].numpy(), int(L), 16)
        mean = ref.widen(v, "f16").mean(axis=0)
        for h in range(8):
            np.testing.assert_allclose(out[i, h], mean[h // 4], atol=2e-3, rtol=0)


# ---------------------------------------------------------------- bitwise invariants on the GPU

def _relabel(W, perm):
    """The same workload with physical block b moved to perm[b]."""
    pool = torch.empty_like(W.pool)
    pool[torch.from_numpy(perm)] = W.pool
    bt = W.block_tables.numpy().copy()
    live = bt >= 0
    bt[live] = perm[bt[live]]
    slots = W.slot_mapping.numpy().copy()
    ok = slots >= 0
    slots[ok] = perm[slots[ok] // 16] * 16 + slots[ok] % 16
    import dataclasses
    return dataclasses.replace(W, pool=pool, block_tables=torch.from_numpy(bt.astype(np.int32)),
                               slot_mapping=torch.from_numpy(slots))


@pytest.mark.parametrize("n", [2, 4])
def test_block_permutation_invariance_bitwise(n):
    spec = wl.SPECS[n]
    small = wl.Spec(spec.name, 12, spec.num_q_heads, spec.num_kv_heads, spec.head_size,
                    spec.q_dtype, spec.kv_dtype,
                    spec.lens if spec.lens[0] != "shared_prefix" else ("shared_prefix", 3, 4, 1024, 256))
    W = wl.make_workload(small, 50 + n)
    a = H.gpu_step(W, H.gpu_pool(W)).cpu()
    perm = np.random.default_rng(n).permutation(W.num_blocks)
    W2 = _relabel(W, perm)
    b = H.gpu_step(W2, H.gpu_pool(W2)).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_equals_private_copies_bitwise():
    spec = wl.Spec("shared", 8, 32, 8, 128, "f16", "f16", ("shared_prefix", 2, 4, 1024, 256))
    W = wl.make_workload(spec, 61)
    a = H.gpu_step(W, H.gpu_pool(W)).cpu()
    # give every sequence private copies of its prefix blocks
    bt = W.block_tables.numpy().copy()
    extra, pool = [], W.pool
    nxt = W.num_blocks
    copies = []
    for i in range(spec.num_seqs):
        for j in range(64):
            copies.append(bt[i, j])
            bt[i, j] = nxt
            nxt += 1
    pool = torch.cat([pool, pool[torch.tensor(copies)]], dim=0)
    import dataclasses
    W2 = dataclasses.replace(W, pool=pool, num_blocks=nxt,
                             block_tables=torch.from_numpy(bt.astype(np.int32)))
    b = H.gpu_step(W2, H.gpu_pool(W2)).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_run_to_run_bitwise_deterministic(n):
    """Repeated decodes of one device state give identical bits, the first run
    after set-up included (a stage refilled by TMA while still being read
    showed up here as a rare, large change in one CTA's partial output)."""
    from paged_kv_cache_296_gb300.runner import DecodeStep
    W = wl.make_workload(wl.SPECS[n], n, device="cuda")
    S = DecodeStep(W, device="cuda")
    S.write()
    torch.cuda.synchronize()
    outs = []
    for _ in range(24):
        S.decode()
        outs.append(S.out.clone())
    ref = outs[0].view(torch.int16)
    bad = [k for k, o in enumerate(outs) if not torch.equal(o.view(torch.int16), ref)]
    assert not bad, f"runs {bad} differ from run 0"
    c, _ = _append_step(W)
    d, _ = _append_step(W)
    assert torch.equal(c.view(torch.int16), d.view(torch.int16))


def test_deterministic_and_split_matches_unsplit():
    W = wl.make_workload(wl.SPECS[3], 3)
    pool = H.gpu_pool(W)
    a = H.gpu_step(W, pool, partition_size=512).cpu()             # up to 8 partitions
    b = H.gpu_step(W, pool, partition_size=512).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    whole = H.gpu_step(W, pool, partition_size=4096).cpu()      # one partition per sequence
    err = (a.float() - whole.float()).abs().max().item()
    assert err <= 1e-2, err


def test_check_tables_counts_bad_indices():
    W = wl.make_workload(wl.SPECS[1], 1, table_garbage=True)
    bt, cl, sm = W.block_tables.cuda(), W.context_lens.cuda(), W.slot_mapping.cuda()
    assert pa.pa_check_tables(bt, cl, sm, W.num_blocks) == [0, 0, 0]
    bt2 = W.block_tables.clone()
    bt2[3, 1] = W.num_blocks          # sequence 3 (17 tokens) uses two blocks
    cl2 = W.context_lens.clone()
    cl2[0] = 10 ** 6
    sm2 = W.slot_mapping.clone()
    sm2[2] = W.num_blocks * 16
    counts = pa.pa_check_tables(bt2.cuda(), cl2.cuda(), sm2.cuda(), W.num_blocks)
    assert counts == [1, 1, 1]


# ---------------------------------------------------------------- fused append + in-kernel merge

def _append_step(W, partition_size=0, workspace=None):
    """pa_decode_append on a fresh device copy of W; returns (out, pool)."""
    from paged_kv_cache_296_gb300.runner import DecodeStep
    S = DecodeStep(W, device="cuda", partition_size=partition_size, shared=False)
    pa.pa_decode_append(S.out, S.q, S.k_new, S.v_new, S.slot_mapping, S.k_cache, S.v_cache,
                        S.block_tables, S.context_lens, S.scale, kv_scale=S.kv_scale,
                        partition_size=partition_size,
                        workspace=S.workspace if workspace is None else workspace)
    return S.out, S.pool


def _separate_step(W, partition_size=0):
    """pa_reshape_and_cache then pa_decode (no shared-prefix groups); returns (out, pool)."""
    from paged_kv_cache_296_gb300.runner import DecodeStep
    S = DecodeStep(W, device="cuda", partition_size=partition_size, shared=False)
    S.write()
    S.decode()
    return S.out, S.pool


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_append_equals_write_then_decode_bitwise(n):
    W = wl.make_workload(wl.SPECS[n], n, device="cuda")
    out_a, pool_a = _append_step(W)
    out_s, pool_s = _separate_step(W)
    assert torch.equal(pool_a.view(torch.uint8), pool_s.view(torch.uint8))
    assert torch.equal(out_a.view(torch.int16), out_s.view(torch.int16))


@pytest.mark.parametrize("seed", range(12))
def test_decode_append_matches_oracle(seed):
    spec = wl.random_spec(200 + seed)
    W = wl.make_workload(spec, 2000 + seed, poison=True, table_garbage=True)
    out, pool = _append_step(W, partition_size=spec.partition_size)
    got = H.widen_out(out, spec.q_dtype)
    assert np.isfinite(got).all(), "the appended token was not visible to the attention"
    g = spec.num_q_heads // spec.num_kv_heads
    if spec.kv_dtype == "e4m3":
        for i in range(spec.num_seqs):
            for h in range(spec.num_kv_heads):
                blocks, mini = H.mini_case(W, i, h)
                opool, want = H.oracle_mini(W, mini)
                gpool = H.bits_of(pool[torch.from_numpy(blocks).cuda()][:, :, :, h:h + 1].cpu())
                live = ~e4m3.is_nan_code(opool)
                assert np.array_equal(gpool[live], opool[live])
                H.assert_close(got[i, h * g:(h + 1) * g], want, spec, f"s{i} h{h}")
    else:
        opool = H.oracle_pool_after_step(W)
        assert np.array_equal(H.bits_of(pool.cpu()), opool)
        H.assert_close(got, H.oracle_decode_full(W, opool), spec, spec.name)


def test_many_partitions_merge():
    # 9000 tokens in 16-token partitions: 563 partials per head to merge.
    spec = wl.Spec("many partitions", 2, 8, 2, 64, "f16", "f16", ("fixed", [9000, 5000]))
    W = wl.make_workload(spec, 91, poison=True)
    _full_check(W, partition_size=16)
    out_small, _ = _separate_step(W, partition_size=16)
    out_big, _ = _separate_step(W, partition_size=512)
    err = (out_small.float() - out_big.float()).abs().max().item()
    assert err <= 2e-3, err


def test_workspace_garbage_does_not_matter():
    # Every partial the merge reads is written earlier in the same call, so
    # whatever the workspace held before (here: random bytes) cannot leak in.
    W = wl.make_workload(wl.SPECS[5], 5, device="cuda")
    from paged_kv_cache_296_gb300.runner import DecodeStep
    S = DecodeStep(W, device="cuda")
    ws_zero = torch.zeros_like(S.workspace)
    ws_junk = torch.randint(0, 256, S.workspace.shape, dtype=torch.uint8, device="cuda")
    S.write()
    outs = []
    for ws in (ws_zero, ws_junk, ws_junk, ws_zero):
        pa.pa_decode(S.out, S.q, S.k_cache, S.v_cache, S.block_tables, S.context_lens, S.scale,
                     kv_scale=S.kv_scale, workspace=ws)
        outs.append(S.out.clone())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("hkv,group,path,part", [(1, 8, "separate", 0), (3, 2, "append", 0),
                                                 (5, 1, "separate", 64), (3, 4, "append", 512),
                                                 (1, 4, "append", 16)])
def test_fp8_odd_kv_head_counts(hkv, group, path, part):
    """E4M3 CTAs take KV heads in pairs; with an odd count the last pair's second
    head does not exist.  Every real head must match the oracle, the pool must
    hold exactly the oracle's bytes, and nothing past ``out`` may be written."""
    lens = [1, 17, 300, 1500, 40, 0]
    spec = wl.Spec("fp8, odd KV head count", len(lens), hkv * group, hkv, 128, "bf16", "e4m3",
                   ("fixed", lens), ("factor", 1.3))
    W = wl.make_workload(spec, 40 + hkv + group, poison=True, table_garbage=True)
    from paged_kv_cache_296_gb300.runner import DecodeStep
    S = DecodeStep(W, device="cuda", partition_size=part)
    n = S.out.numel()
    canary = torch.full((n + 4096,), -7.0, dtype=S.out.dtype, device="cuda")
    out = canary[:n].view(S.out.shape)
    if path == "append":
        pa.pa_decode_append(out, S.q, S.k_new, S.v_new, S.slot_mapping, S.k_cache, S.v_cache,
                            S.block_tables, S.context_lens, S.scale, kv_scale=S.kv_scale,
                            partition_size=part, workspace=S.workspace)
    else:
        S.write()
        pa.pa_decode(out, S.q, S.k_cache, S.v_cache, S.block_tables, S.context_lens, S.scale,
                     kv_scale=S.kv_scale, partition_size=part, workspace=S.workspace)
    assert bool((canary[n:] == -7.0).all()), "a write landed past the output"
    got = H.widen_out(out, spec.q_dtype)
    assert np.isfinite(got).all()
    assert np.array_equal(got[-1], np.zeros_like(got[-1])), "empty context must give zeros"
    for i in range(spec.num_seqs):
        for h in range(hkv):
            blocks, mini = H.mini_case(W, i, h)
            opool, want = H.oracle_mini(W, mini)
            if len(blocks):
                gpool = H.bits_of(S.pool[torch.from_numpy(blocks).cuda()][:, :, :, h:h + 1].cpu())
                live = ~e4m3.is_nan_code(opool)
                assert np.array_equal(gpool[live], opool[live])
            H.assert_close(got[i, h * group:(h + 1) * group], want, spec, f"s{i} h{h}")


def test_very_long_context_balanced_split():
    """One 131072-token sequence (8192 blocks) beside three short ones: the
    balanced split gives the long one most of the wave's CTAs and the merge
    folds their partials.  Every output against the oracle."""
    lens = [131072, 1, 700, 33]
    spec = wl.Spec("very long context", len(lens), 8, 2, 128, "f16", "f16", ("fixed", lens),
                   ("factor", 1.05))
    W = wl.make_workload(spec, 88, poison=True, table_garbage=True)
    assert pa.pa_decode_partition_size(len(lens), 2, W.max_blocks_per_seq) == 0  # balanced
    _full_check(W)


@pytest.mark.parametrize("kv,q", [("f16", "f16"), ("e4m3", "bf16")])
def test_largest_batch_sampled(kv, q):
    """The largest batch the calls take (65535 sequences of 0-39 tokens, two KV
    heads): a grid of one CTA per (sequence, KV head group).  Every output is
    finite; the first, the last and 200 random sequences match the oracle."""
    B = 65535
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 40, B)]
    spec = wl.Spec("largest batch", B, 4, 2, 64, q, kv, ("fixed", lens), ("factor", 1.2))
    W = wl.make_workload(spec, 77, poison=True)
    pool = H.gpu_pool(W)
    out = H.gpu_step(W, pool)
    got = H.widen_out(out, q)
    assert np.isfinite(got).all(), "NaN/inf output: a poisoned slot was read"
    for i in sorted({0, 1, B - 1} | {int(x) for x in rng.integers(0, B, 200)}):
        for h in range(2):
            _, mini = H.mini_case(W, i, h)
            _, want = H.oracle_mini(W, mini)
            H.assert_close(got[i, 2 * h:2 * h + 2], want, spec, f"seq {i} kv head {h}")
    assert pa.pa_device_status(clear=True) == 0


@pytest.mark.parametrize("num_seqs", [1, 31, 32, 33, 100])
def test_balanced_split_batch_sizes(num_seqs):
    """Few (sequence, KV head) pairs: the kernel plans a balanced split from the
    lengths (one warp up to 32 sequences, all warps above).  Every output must
    match the oracle, including empty and one-token sequences."""
    rng = np.random.default_rng(num_seqs)
    lens = [int(x) for x in np.exp(rng.uniform(0, np.log(6000), num_seqs))]
    if num_seqs == 1:
        lens = [5000]
    else:
        lens[0], lens[1] = 0, 1
        lens[-1] = 5000
    spec = wl.Spec("balanced split", num_seqs, 8, 2, 64, "f16", "f16", ("fixed", lens),
                   ("factor", 1.2))
    W = wl.make_workload(spec, 500 + num_seqs, poison=True, table_garbage=True)
    assert pa.pa_decode_partition_size(num_seqs, 2, W.max_blocks_per_seq) == 0  # balanced
    _full_check(W)
