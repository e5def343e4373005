"""Pins for the oracle's block manager (CPU only).

Checked against the pages' own sketch (blocks taken from the front of a free
list that starts as every id in order, ceil(n / block_size) blocks per
sequence, an out-of-memory error when it runs dry), invariants (reference
counts equal table occurrences, free and used blocks partition the pool) and a
memory model: random allocate / append / fork / free sequences write token
values through the returned slots (after the returned copy-on-write copies),
and every sequence gathered through its block table must read back exactly its
own logical tokens.
"""

import random

import pytest

from oracle.block_manager import BlockManager, OutOfBlocks


def test_pages_sketch_allocation_order_and_ceil():
    bm = BlockManager(8)
    bm.allocate("a", 40)          # ceil(40 / 16) = 3 blocks, from the front
    bm.allocate("b", 16)
    bm.allocate("c", 1)
    assert bm.tables == {"a": [0, 1, 2], "b": [3], "c": [4]}
    bm.allocate("d", 0)
    assert bm.tables["d"] == [] and bm.num_free() == 3


def test_out_of_blocks_changes_nothing():
    bm = BlockManager(4)
    bm.allocate("a", 40)
    with pytest.raises(OutOfBlocks):
        bm.allocate("b", 20)      # needs 2, 1 free
    assert "b" not in bm.tables and bm.num_free() == 1
    with pytest.raises(OutOfBlocks):
        bm.append("a", 30)        # 40 + 30 = 70 tokens -> 5 blocks, 2 more needed
    assert bm.lens["a"] == 40 and bm.tables["a"] == [0, 1, 2]


def test_append_takes_a_block_when_the_last_one_is_full():
    bm = BlockManager(4)
    bm.allocate("a", 15)
    slots, copies = bm.append("a", 1)       # fills block 0
    assert slots == [15] and copies == [] and bm.tables["a"] == [0]
    slots, copies = bm.append("a", 2)       # spills into a new block
    assert slots == [16, 17] and bm.tables["a"] == [0, 1]


def test_release_order_and_reuse():
    bm = BlockManager(6)
    bm.allocate("a", 48)                    # [0, 1, 2]
    bm.allocate("b", 16)                    # [3]
    bm.free_seq("a")                        # free list: 4, 5, 0, 1, 2
    bm.allocate("c", 40)
    assert bm.tables["c"] == [4, 5, 0]


def test_fork_shares_and_copy_on_write_on_a_partial_shared_block():
    bm = BlockManager(8)
    bm.allocate("p", 20)                    # [0, 1], block 1 holds 4 tokens
    bm.fork("p", "c")
    assert bm.ref[0] == 2 and bm.ref[1] == 2
    slots, copies = bm.append("c", 1)       # position 20 is in the shared block 1
    assert copies == [(1, 2)] and bm.tables["c"] == [0, 2] and slots == [2 * 16 + 4]
    assert bm.ref[1] == 1 and bm.ref[2] == 1
    slots, copies = bm.append("p", 1)       # block 1 is now the parent's alone
    assert copies == [] and slots == [1 * 16 + 4]
    bm.fork("p", "q")                       # 21 tokens: full block 0 + 5 in block 1
    bm.free_seq("p")
    assert bm.ref[0] == 2 and bm.ref[1] == 1   # still held by c (block 0) and q


def test_full_shared_block_needs_no_copy():
    bm = BlockManager(8)
    bm.allocate("p", 32)                    # two full blocks
    bm.fork("p", "c")
    slots, copies = bm.append("c", 3)
    assert copies == [] and bm.tables["c"] == [0, 1, 2] and slots == [32, 33, 34]


def _check_invariants(bm):
    count = [0] * bm.num_blocks
    for t in bm.tables.values():
        for b in t:
            count[b] += 1
    assert count == bm.ref
    used = {b for b in range(bm.num_blocks) if bm.ref[b] > 0}
    free = list(bm.free)
    assert len(free) == len(set(free)) and not (used & set(free))
    assert len(used) + len(free) == bm.num_blocks
    for s, t in bm.tables.items():
        assert len(t) == bm.blocks_for(bm.lens[s])


@pytest.mark.parametrize("seed", range(30))
def test_memory_model_random_operations(seed):
    rnd = random.Random(seed)
    bs = 16
    bm = BlockManager(rnd.choice([6, 12, 40]), bs)
    pool = {}        # slot -> token value (the cache, per slot)
    logical = {}     # seq -> the tokens it holds, in order
    next_val = [1]

    def write(seq, slots):
        vals = []
        for s in slots:
            pool[s] = next_val[0]
            vals.append(next_val[0])
            next_val[0] += 1
        logical[seq].extend(vals)

    def copy(copies):
        for src, dst in copies:
            for o in range(bs):
                if src * bs + o in pool:
                    pool[dst * bs + o] = pool[src * bs + o]

    ids = 0
    for _ in range(200):
        op = rnd.random()
        live = list(bm.tables)
        try:
            if op < 0.25 or not live:
                n = rnd.randint(0, 50)
                bm.allocate(ids, n)
                logical[ids] = []
                write(ids, [bm.tables[ids][p // bs] * bs + p % bs for p in range(n)])
                ids += 1
            elif op < 0.6:
                s = rnd.choice(live)
                slots, copies = bm.append(s, rnd.randint(1, 20))
                copy(copies)
                write(s, slots)
            elif op < 0.8:
                s = rnd.choice(live)
                bm.fork(s, ids)
                logical[ids] = list(logical[s])
                ids += 1
            else:
                s = rnd.choice(live)
                bm.free_seq(s)
                del logical[s]
        except OutOfBlocks:
            pass
        _check_invariants(bm)
        for s, t in bm.tables.items():
            L = bm.lens[s]
            got = [pool.get(t[p // bs] * bs + p % bs) for p in range(L)]
            assert got == logical[s], f"seq {s}"


# ---------------------------------------------------------------- prefix caching

def _toks(*runs):
    out = []
    for start, n in runs:
        out += list(range(start, start + n))
    return out


def test_prefix_hits_for_a_shared_system_prompt():
    bm = BlockManager(32)
    system = _toks((1000, 40))                      # 2 full blocks + 8 tokens
    a = system + _toks((1, 30))
    b = system + _toks((500, 25))
    assert bm.allocate_cached("a", a) == 0
    assert bm.allocate_cached("b", b) == 32          # the 2 full system blocks
    assert bm.tables["b"][:2] == bm.tables["a"][:2]
    assert bm.tables["b"][2] != bm.tables["a"][2]    # the block mixing prompts differs
    assert bm.ref[bm.tables["a"][0]] == 2


def test_cached_blocks_survive_release_until_handed_out_again():
    bm = BlockManager(8)
    p = _toks((7, 48))                               # 3 full blocks
    bm.allocate_cached("a", p)
    held = list(bm.tables["a"])
    bm.free_seq("a")
    assert bm.allocate_cached("b", p + [1]) == 48    # all three reused from the free list
    assert bm.tables["b"][:3] == held
    bm.free_seq("b")
    bm.allocate("x", 8 * 16 - 16)                    # takes 7 blocks: evicts cached ones
    bm.free_seq("x")
    assert bm.allocate_cached("c", p + [1]) < 48


def test_a_fully_cached_prompt_still_computes_its_last_block():
    bm = BlockManager(8)
    p = _toks((3, 32))
    bm.allocate_cached("a", p)
    assert bm.allocate_cached("b", p) == 16          # not 32: one block is recomputed
    assert bm.allocate_cached("c", p[:31]) == 16


def test_a_reused_parent_id_does_not_match_old_children():
    # Block 0 (the first block of prompt p) is handed out again for other
    # content X while block 1 (p's second block, keyed under block 0's old
    # generation) is still cached.  A prompt X + p's second block must not
    # pick up block 1: its K/V were computed after p's first block, not X's.
    bm = BlockManager(4)
    p = _toks((100, 33))                             # blocks 0, 1 full, 2 partial
    bm.allocate_cached("a", p)
    bm.free_seq("a")                                 # free list: 3, 0, 1, 2
    bm.allocate("x", 16)                             # takes 3
    X = _toks((9, 16))
    assert bm.allocate_cached("y", X) == 0           # takes 0 (evicted), registers X there
    assert bm.tables["y"] == [0]
    z = X + p[16:32] + [5]
    assert bm.allocate_cached("z", z) == 16          # block 0 hits; block 1 must not


@pytest.mark.parametrize("seed", range(20))
def test_prefix_cache_memory_model(seed):
    # The K/V a slot holds stands for the token prefix that produced it; every
    # sequence read back through its table must see its own prefixes.
    rnd = random.Random(1000 + seed)
    bs = 16
    bm = BlockManager(rnd.choice([10, 24, 64]), bs)
    pool = {}
    seqs = {}    # seq -> its token list
    bases = [_toks((rnd.randint(0, 5) * 100, rnd.randint(0, 70))) for _ in range(4)]
    nid = 0
    for _ in range(150):
        op = rnd.random()
        live = list(bm.tables)
        try:
            if op < 0.45 or not live:
                toks = list(rnd.choice(bases)) + _toks((rnd.randint(0, 3) * 7, rnd.randint(0, 40)))
                if rnd.random() < 0.3:
                    toks = toks[:rnd.randint(0, len(toks))]
                cached = bm.allocate_cached(nid, toks)
                assert cached % bs == 0 and (cached < len(toks) or len(toks) == 0)
                t = bm.tables[nid]
                for pos in range(cached, len(toks)):         # compute only what is not cached
                    pool[t[pos // bs] * bs + pos % bs] = tuple(toks[:pos + 1])
                seqs[nid] = toks
                nid += 1
            elif op < 0.7:
                s = rnd.choice(live)
                extra = _toks((rnd.randint(0, 9) * 11, rnd.randint(1, 20)))
                slots, copies = bm.append(s, len(extra))
                for src, dst in copies:
                    for o in range(bs):
                        if src * bs + o in pool:
                            pool[dst * bs + o] = pool[src * bs + o]
                base = len(seqs[s])
                seqs[s] = seqs[s] + extra
                for k, sl in enumerate(slots):
                    pool[sl] = tuple(seqs[s][:base + k + 1])
                if rnd.random() < 0.5:
                    bm.register(s, seqs[s])
            elif op < 0.8:
                s = rnd.choice(live)
                bm.fork(s, nid)
                seqs[nid] = list(seqs[s])
                nid += 1
            else:
                s = rnd.choice(live)
                bm.free_seq(s)
                del seqs[s]
        except OutOfBlocks:
            pass
        _check_invariants(bm)
        for s, t in bm.tables.items():
            toks = seqs[s]
            for pos in range(len(toks)):
                assert pool.get(t[pos // bs] * bs + pos % bs) == tuple(toks[:pos + 1]), (s, pos)
