"""GPU parity of the shared-prefix decode (pa_decode_shared, pa_decode_append_shared).

Groups of sequences whose block tables begin with the same physical blocks
(parallel sampling: "vLLM GitHub 项目…", section 二 item 4) are decoded with
each shared block read once for the whole group.  The result must be the
attention the tables define, checked against the float64 oracle on the same
tables, with every unread slot of the pool poisoned with NaN.

Shared workloads are built from a seeded workload by pointing the first P
entries of every member's table at the group leader's blocks (all of them
full of live tokens); a member whose context ends inside those P blocks gets
no new token (its slot would lie in a shared block) and attends only its own
length.
"""

import numpy as np
import pytest
import torch

from oracle import e4m3
from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300 import workloads as wl
from paged_kv_cache_296_gb300.workloads import BLOCK_SIZE

import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    pa.load()
    pa.pa_device_status(clear=True)
    yield
    assert pa.pa_device_status(clear=True) == 0


def alias_groups(W, groups, rng):
    """Make each group's members share the leader's first P blocks.

    ``groups``: list of member lists (first = leader).  Returns the group
    arrays (CPU SharedGroups) with P per group: a random count of the
    leader's full, live blocks (its last token, the one the step writes, is
    never inside them)."""
    tables = W.block_tables.clone()
    slots = W.slot_mapping.clone()
    lens = W.context_lens
    offs, seqs, blks = [0], [], []
    for mem in groups:
        lead = mem[0]
        full = (int(lens[lead]) - 1) // BLOCK_SIZE
        P = int(rng.integers(1, full + 1)) if full >= 1 else 0
        if P == 0:
            continue
        for s in mem[1:]:
            tables[s, :P] = tables[lead, :P]
            if int(lens[s]) <= P * BLOCK_SIZE:
                slots[s] = -1      # its new token would land in a shared block
        seqs += mem
        offs.append(len(seqs))
        blks.append(P)
    W.block_tables = tables.contiguous()
    W.slot_mapping = slots
    return pa.SharedGroups(torch.tensor(offs, dtype=torch.int32),
                           torch.tensor(seqs or [0], dtype=torch.int32),
                           torch.tensor(blks or [0], dtype=torch.int32))


def run_shared(W, groups, pool, path, workspace=None):
    """One step on the GPU through the shared-prefix calls; returns out."""
    dev = pool.device
    kc, vc = pa.kv_views(pool)
    g = groups.to(dev)
    out = torch.empty(W.q.shape, dtype=W.q.dtype, device=dev)
    args = (W.block_tables.to(dev), W.context_lens.to(dev), W.scale, g)
    if path == "append":
        pa.pa_decode_append_shared(out, W.q.to(dev), W.k_new.to(dev), W.v_new.to(dev),
                                   W.slot_mapping.to(dev), kc, vc, *args, kv_scale=W.kv_scale,
                                   workspace=workspace)
    else:
        pa.pa_reshape_and_cache(W.k_new.to(dev), W.v_new.to(dev), kc, vc, W.slot_mapping.to(dev),
                                kv_scale=W.kv_scale)
        pa.pa_decode_shared(out, W.q.to(dev), kc, vc, *args, kv_scale=W.kv_scale,
                            workspace=workspace)
    return out


def check_against_oracle(W, pool, out, what):
    spec = W.spec
    got = H.widen_out(out, spec.q_dtype)
    assert np.isfinite(got).all(), "NaN/inf output: a poisoned slot was read"
    if spec.kv_dtype != "e4m3":
        opool = H.oracle_pool_after_step(W)
        assert np.array_equal(H.bits_of(pool.cpu()), opool), "pool after the write differs"
        H.assert_close(got, H.oracle_decode_full(W, opool), spec, what)
        return
    g = spec.num_q_heads // spec.num_kv_heads
    for i in range(spec.num_seqs):
        for h in range(spec.num_kv_heads):
            blocks, mini = H.mini_case(W, i, h)
            opool, want = H.oracle_mini(W, mini)
            if len(blocks):
                gp = H.bits_of(pool[torch.from_numpy(blocks).cuda()][:, :, :, h:h + 1].cpu())
                live = ~e4m3.is_nan_code(opool)
                assert np.array_equal(gp[live], opool[live]), f"{what}: pool s{i} h{h}"
            H.assert_close(got[i, h * g:(h + 1) * g], want, spec, f"{what} s{i} h{h}")


def random_shared_case(seed, kv=None):
    rng = np.random.default_rng(seed)
    d = int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 3]))
    kvd = kv or str(rng.choice(["f16", "bf16", "e4m3"]))
    qd = kvd if kvd != "e4m3" else str(rng.choice(["f16", "bf16"]))
    B = int(rng.integers(2, 14))
    lens = [int(x) for x in rng.integers(0, 700, B)]
    lens[0] = max(lens[0], 40)
    spec = wl.Spec(f"shared seed {seed}", B, hkv * G, hkv, d, qd, kvd, ("fixed", lens),
                   ("factor", 1.5))
    W = wl.make_workload(spec, 3000 + seed, poison=True, table_garbage=True)
    order = [int(x) for x in rng.permutation(B)]
    groups, i = [], 0
    while i < B:
        k = int(rng.integers(1, 7))
        mem = [s for s in order[i:i + k] if lens[s] > 0]
        i += k
        if len(mem) >= 2:
            # the leader: a member with the longest context
            mem.sort(key=lambda s: -lens[s])
            groups.append(mem)
    return W, alias_groups(W, groups, rng)


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("path", ["append", "separate"])
def test_shared_prefix_workload_all_outputs(path):
    """16 prompts x 8 samples, 1024-token prefix: every output against the oracle."""
    W = wl.make_workload(wl.SPECS[4], 4, poison=True)
    groups = pa.pa_find_shared_prefixes(W.block_tables, W.context_lens, 32, 8)
    assert groups.num_groups == 16
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, path)
    check_against_oracle(W, pool, out, f"shared prefix, {path}")


@pytest.mark.parametrize("seed", H.seeds(16))
def test_shared_random_shapes(seed):
    W, groups = random_shared_case(seed)
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, "append" if seed % 2 else "separate")
    check_against_oracle(W, pool, out, W.spec.name)


@pytest.mark.parametrize("kv,q", [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16")])
def test_members_shorter_than_the_shared_blocks(kv, q):
    """Members whose contexts end inside the group's shared blocks (one of them
    empty) attend only their own tokens; the others continue past them."""
    lens = [900, 100, 33, 0, 640, 17, 1000]
    spec = wl.Spec("short members", len(lens), 16, 4, 128, q, kv, ("fixed", lens),
                   ("factor", 1.4))
    W = wl.make_workload(spec, 71, poison=True, table_garbage=True)
    tables = W.block_tables.clone()
    slots = W.slot_mapping.clone()
    P = 40                                   # 640 tokens of sequence 6's blocks
    for s in range(6):
        tables[s, :P] = tables[6, :P]
        if lens[s] <= P * BLOCK_SIZE:
            slots[s] = -1
    W.block_tables, W.slot_mapping = tables.contiguous(), slots
    groups = pa.SharedGroups(torch.tensor([0, 7], dtype=torch.int32),
                             torch.tensor([6, 0, 1, 2, 3, 4, 5], dtype=torch.int32),
                             torch.tensor([P], dtype=torch.int32))
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, "append")
    check_against_oracle(W, pool, out, "short members")
    assert np.array_equal(H.widen_out(out, q)[3], np.zeros((16, 128))), "empty context: zeros"


def test_groups_larger_than_the_mma_columns():
    """G = 8: a prefix tile holds 4 members per KV head; members past that are
    decoded as unshared sequences and must still be right."""
    lens = [500, 480, 460, 440, 420, 400, 380]
    spec = wl.Spec("big group", len(lens), 16, 2, 64, "f16", "f16", ("fixed", lens),
                   ("factor", 1.3))
    W = wl.make_workload(spec, 72, poison=True)
    groups = alias_groups(W, [list(range(7))], np.random.default_rng(3))
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, "append")
    check_against_oracle(W, pool, out, "big group")


@pytest.mark.parametrize("hkv,group", [(1, 8), (3, 2), (5, 1)])
def test_fp8_shared_odd_kv_head_counts(hkv, group):
    lens = [1500, 1400, 300, 1499, 17, 0, 800]
    spec = wl.Spec("fp8 shared, odd KV heads", len(lens), hkv * group, hkv, 128, "bf16", "e4m3",
                   ("fixed", lens), ("factor", 1.3))
    W = wl.make_workload(spec, 80 + hkv, poison=True, table_garbage=True)
    groups = alias_groups(W, [[0, 1, 3], [2, 6, 4]], np.random.default_rng(hkv))
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, "append")
    check_against_oracle(W, pool, out, "fp8 shared odd heads")


@pytest.mark.parametrize("kv,q", [("f16", "f16"), ("e4m3", "bf16")])
def test_plan_at_its_size_limit(kv, q):
    """The largest batch the stream-K plan holds: 1024 sequences in 512 groups of
    two (short contexts keep the oracle quick).  Every output against the oracle."""
    rng = np.random.default_rng(91)
    B = 1024
    lens = [int(x) for x in rng.integers(20, 200, B)]
    spec = wl.Spec("plan size limit", B, 4, 2, 64, q, kv, ("fixed", lens), ("factor", 1.3))
    W = wl.make_workload(spec, 91, poison=True, table_garbage=True)
    order = [int(x) for x in rng.permutation(B)]
    pairs = [sorted(order[i:i + 2], key=lambda s: -lens[s]) for i in range(0, B, 2)]
    groups = alias_groups(W, pairs, rng)
    assert groups.num_groups >= 400
    pool = H.gpu_pool(W)
    out = run_shared(W, groups, pool, "append")
    check_against_oracle(W, pool, out, f"plan size limit, {kv}")


def test_plan_past_its_size_limit_is_refused():
    """One sequence more than the plan holds: refused before any launch."""
    B = 1025
    spec = wl.Spec("past the plan", B, 4, 2, 64, "f16", "f16", ("fixed", [40] * B))
    W = wl.make_workload(spec, 92, device="cuda")
    groups = pa.SharedGroups(torch.tensor([0, 2], dtype=torch.int32, device="cuda"),
                             torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                             torch.tensor([1], dtype=torch.int32, device="cuda"))
    kc, vc = pa.kv_views(H.gpu_pool(W))
    out = torch.empty_like(W.q)
    with pytest.raises(pa.PagedAttentionError, match="at most 1024 sequences"):
        pa.pa_decode_shared(out, W.q, kc, vc, W.block_tables, W.context_lens, W.scale, groups)
    assert pa.pa_device_status(clear=True) == 0


# ---------------------------------------------------------------- bitwise properties

def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t


@pytest.mark.parametrize("config", [4, 5])
def test_append_equals_write_then_decode_bitwise(config):
    W = wl.make_workload(wl.SPECS[config], config, device="cuda")
    groups = pa.pa_find_shared_prefixes(W.block_tables, W.context_lens, W.spec.num_q_heads,
                                        W.spec.num_kv_heads)
    if config == 5:   # no shared tables: let the first two sequences share 100 blocks
        W.block_tables = W.block_tables.cpu()
        W.slot_mapping = W.slot_mapping.cpu()
        groups = alias_groups(W, [[0, 1]], np.random.default_rng(5))
        W.block_tables = W.block_tables.cuda()
        W.slot_mapping = W.slot_mapping.cuda()
    pool_a = H.gpu_pool(W)
    pool_s = pool_a.clone()
    out_a = run_shared(W, groups, pool_a, "append")
    out_s = run_shared(W, groups, pool_s, "separate")
    assert torch.equal(pool_a, pool_s)
    assert torch.equal(_bits(out_a), _bits(out_s))


def test_shared_run_to_run_bitwise_and_workspace_garbage():
    W = wl.make_workload(wl.SPECS[4], 4, device="cuda")
    groups = pa.pa_find_shared_prefixes(W.block_tables, W.context_lens, 32, 8).to("cuda")
    pool = H.gpu_pool(W)
    kc, vc = pa.kv_views(pool)
    pa.pa_reshape_and_cache(W.k_new, W.v_new, kc, vc, W.slot_mapping)
    nbytes = pa.pa_decode_shared_workspace_size(128, 32, 8, 128, W.max_blocks_per_seq, 16,
                                                groups.num_groups)
    ws_junk = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda")
    ws_nan = torch.full((nbytes // 4,), float("nan"), device="cuda").view(torch.uint8)
    outs = []
    for ws in (ws_junk, ws_nan, ws_junk, ws_nan, ws_junk):
        out = torch.empty_like(W.q)
        pa.pa_decode_shared(out, W.q, kc, vc, W.block_tables, W.context_lens, W.scale, groups,
                            workspace=ws)
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(_bits(o), _bits(outs[0]))


def test_no_groups_is_pa_decode_bitwise():
    """With no groups the shared call is pa_decode with the library's choice of
    split: the same kernels and plan, the same bits."""
    W = wl.make_workload(wl.SPECS[5], 5, device="cuda")
    assert pa.pa_decode_partition_size(8, 8, W.max_blocks_per_seq) == 0
    pool = H.gpu_pool(W)
    kc, vc = pa.kv_views(pool)
    none = pa.SharedGroups(torch.zeros(1, dtype=torch.int32, device="cuda"),
                           torch.zeros(1, dtype=torch.int32, device="cuda"),
                           torch.zeros(1, dtype=torch.int32, device="cuda"))
    a, b = torch.empty_like(W.q), torch.empty_like(W.q)
    pa.pa_decode(a, W.q, kc, vc, W.block_tables, W.context_lens, W.scale, kv_scale=W.kv_scale)
    pa.pa_decode_shared(b, W.q, kc, vc, W.block_tables, W.context_lens, W.scale, none,
                        kv_scale=W.kv_scale)
    assert torch.equal(_bits(a), _bits(b))


def test_shared_matches_unshared_within_tolerance():
    """The same tables decoded without groups (each sample reads the prefix
    itself) and with them agree within the stated tolerance."""
    W = wl.make_workload(wl.SPECS[4], 4, device="cuda")
    groups = pa.pa_find_shared_prefixes(W.block_tables, W.context_lens, 32, 8)
    pool = H.gpu_pool(W)
    kc, vc = pa.kv_views(pool)
    plain = torch.empty_like(W.q)
    pa.pa_decode(plain, W.q, kc, vc, W.block_tables, W.context_lens, W.scale)
    shared = torch.empty_like(W.q)
    pa.pa_decode_shared(shared, W.q, kc, vc, W.block_tables, W.context_lens, W.scale,
                        groups.to("cuda"))
    err = (plain.float() - shared.float()).abs().max().item()
    assert err <= H.ATOL["f16"], err
