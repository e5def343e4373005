"""pa_find_shared_prefixes: the host-side grouping of sequences whose block
tables start with the same physical blocks (no GPU needed).

Sequences forked from one prompt hold its blocks at the start of their tables
("vLLM GitHub 项目…", section 二 item 4); the decode reads those blocks once
per group.  The rule checked here: group by the first table entry, in index
order, at most 32 / G members per group; a group shares the leading entries
equal in every member's table within each member's own ceil(L / 16) blocks;
groups of one, or sharing fewer than min_blocks blocks, are dropped.
"""

import pytest
import torch

from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_296_gb300 import build
    build()
    pa.load()


def _groups(tables, lens, hq=32, hkv=8, min_blocks=1):
    t = torch.tensor(tables, dtype=torch.int32).reshape(len(lens), -1) if lens else \
        torch.zeros((0, 4), dtype=torch.int32)
    g = pa.pa_find_shared_prefixes(t, torch.tensor(lens, dtype=torch.int32).reshape(-1), hq, hkv,
                                   min_blocks)
    offs = g.offsets.tolist()
    return [(g.seqs[offs[k]:offs[k + 1]].tolist(), int(g.blocks[k])) for k in range(g.num_groups)]


def test_shared_prefix_workload_groups():
    # 16 prompts x 8 samples sharing a 1024-token (64-block) prefix
    W = wl.make_workload(wl.SPECS[4], 4)
    got = _groups(W.block_tables.tolist(), W.context_lens.tolist())
    assert len(got) == 16
    seen = []
    for mem, blocks in got:
        assert len(mem) == 8 and blocks == 64
        assert len({m // 8 for m in mem}) == 1          # the samples of one prompt
        seen += mem
    assert sorted(seen) == list(range(128))


def test_group_size_cap_and_order():
    # G = 8 query heads per KV head: 32 / 8 = 4 members per group
    t = [[7, 8, 9]] * 10
    got = _groups(t, [48] * 10, hq=64, hkv=8)
    assert got == [([0, 1, 2, 3], 3), ([4, 5, 6, 7], 3), ([8, 9], 3)]
    # G = 1: up to 32 members
    assert _groups(t, [48] * 10, hq=8, hkv=8) == [(list(range(10)), 3)]


def test_shared_length_is_common_prefix_within_lengths():
    t = [[5, 6, 7, 8], [5, 6, 9, 10], [5, 6, 7, 11], [1, 2, 3, 4]]
    # members 0..2 agree on 2 entries; member 3 starts elsewhere and is alone
    assert _groups(t, [64, 64, 64, 64]) == [([0, 1, 2], 2)]
    # only entries within every member's own ceil(L / 16) blocks count: 20 tokens
    # are 2 blocks (both shared), 10 tokens one
    assert _groups(t, [64, 20, 64, 64]) == [([0, 1, 2], 2)]
    assert _groups(t, [64, 10, 64, 64]) == [([0, 1, 2], 1)]
    # min_blocks drops groups that share too little
    assert _groups(t, [64, 64, 64, 64], min_blocks=3) == []


def test_singletons_and_empty_sequences_are_not_grouped():
    t = [[3, 4], [3, 5], [9, 9], [3, 4]]
    # sequence 1 is empty: it holds no block, so it cannot share one
    assert _groups(t, [32, 0, 32, 32]) == [([0, 3], 2)]
    assert _groups([[1], [2]], [16, 16]) == []
    assert _groups([], []) == []


def test_rejects_bad_arguments():
    lib = pa.load()
    assert lib.pa_find_shared_prefixes(None, None, -1, 4, 16, 8, 8, 1, None, None, None, None) == 1
