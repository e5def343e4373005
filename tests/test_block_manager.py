"""The native block manager (pa_bm_*) against the oracle's model (CPU only).

Both follow the same policy, so every observable result must be identical:
block tables, lengths, the slots an append returns, the copy-on-write pairs,
free-block counts, reference counts and which requests run out of blocks.
"""

import random

import pytest
import torch

from oracle.block_manager import BlockManager as RefManager, OutOfBlocks as RefOOM
from paged_kv_cache_296_gb300 import binding as pa


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_296_gb300 import build
    build()
    return pa.load()


def _same_state(bm, ref):
    assert bm.num_free() == ref.num_free()
    for b in range(ref.num_blocks):
        assert bm.ref_count(b) == ref.ref[b], f"block {b}"
    ids = sorted(ref.tables)
    if not ids:
        return
    width = max(1, max(len(t) for t in ref.tables.values()))
    tables, lens = bm.block_tables(ids, width)
    for k, s in enumerate(ids):
        assert tables[k].tolist() == ref.block_table(s, width), f"seq {s}"
        assert int(lens[k]) == ref.lens[s]


@pytest.mark.parametrize("seed", range(25))
def test_native_manager_matches_the_oracle(lib, seed):
    rnd = random.Random(seed)
    nblocks = rnd.choice([5, 16, 64])
    bm = pa.BlockManager(nblocks)
    ref = RefManager(nblocks)
    next_id = 0
    for _ in range(300):
        live = sorted(ref.tables)
        op = rnd.random()
        if op < 0.2 or not live:
            n = rnd.randint(0, 60)
            exp_oom = False
            try:
                ref.allocate(next_id, n)
            except RefOOM:
                exp_oom = True
            if exp_oom:
                with pytest.raises(pa.OutOfBlocks):
                    bm.allocate(next_id, n)
            else:
                bm.allocate(next_id, n)
            next_id += 1
        elif op < 0.55:
            k = rnd.randint(1, min(4, len(live)))
            seqs = rnd.sample(live, k)
            counts = [rnd.randint(0, 20) for _ in seqs]
            # the oracle applies the batch as one request: all or nothing
            snapshot = (list(ref.free), list(ref.ref), {s: list(t) for s, t in ref.tables.items()},
                        dict(ref.lens))
            want_slots, want_copies, oom = [], [], False
            try:
                for s, c in zip(seqs, counts):
                    sl, cp = ref.append(s, c)
                    want_slots += sl
                    want_copies += cp
            except RefOOM:
                oom = True
                from collections import deque
                ref.free = deque(snapshot[0])
                ref.ref = snapshot[1]
                ref.tables = snapshot[2]
                ref.lens = snapshot[3]
            if oom:
                with pytest.raises(pa.OutOfBlocks):
                    bm.append_batch(seqs, counts)
            else:
                slots, copies = bm.append_batch(seqs, counts)
                assert slots == want_slots
                assert copies == want_copies
        elif op < 0.75:
            s = rnd.choice(live)
            ref.fork(s, next_id)
            bm.fork(s, next_id)
            next_id += 1
        else:
            s = rnd.choice(live)
            ref.free_seq(s)
            bm.free(s)
        _same_state(bm, ref)


def test_errors_change_nothing(lib):
    bm = pa.BlockManager(4)
    bm.allocate(1, 40)
    with pytest.raises(pa.OutOfBlocks):
        bm.allocate(2, 40)
    with pytest.raises(pa.PagedAttentionError):
        bm.allocate(1, 1)                   # id already present
    with pytest.raises(pa.PagedAttentionError):
        bm.append(7, 1)                     # unknown id
    with pytest.raises(pa.PagedAttentionError):
        bm.append_batch([1, 1], [1, 1])     # the same id twice in one batch
    with pytest.raises(pa.PagedAttentionError):
        bm.fork(1, 1)
    with pytest.raises(pa.PagedAttentionError):
        bm.block_tables([1], 2)             # 3 blocks do not fit in width 2
    assert bm.num_free() == 1
    t, lens = bm.block_tables([1], 3)
    assert t.tolist() == [[0, 1, 2]] and lens.tolist() == [40]


def test_a_failed_batch_leaves_its_ids_usable(lib):
    # A batch that fails after naming some sequences (here: an unknown id
    # last) changes nothing, and the same sequences append normally next;
    # a forked child and its parent may appear in one batch.
    bm = pa.BlockManager(16)
    bm.allocate(1, 10)
    bm.allocate(2, 20)
    with pytest.raises(pa.PagedAttentionError):
        bm.append_batch([1, 2, 9], [1, 1, 1])
    assert bm.block_tables([1, 2], 2)[1].tolist() == [10, 20]
    slots, copies = bm.append_batch([1, 2], [1, 1])
    assert slots == [10, 2 * 16 + 4] and copies == []   # seq 2 holds blocks 1 and 2
    bm.fork(1, 3)
    slots, copies = bm.append_batch([3, 1], [1, 1])
    assert copies == [(0, 3)]                # the child copies the shared partial block
    assert slots == [3 * 16 + 11, 11]         # and the parent keeps block 0
    with pytest.raises(pa.PagedAttentionError):
        bm.append_batch([2, 3, 2], [1, 1, 1])


def test_batch_that_does_not_fit_changes_nothing(lib):
    bm = pa.BlockManager(6)
    bm.allocate(1, 16)
    bm.allocate(2, 16)
    with pytest.raises(pa.OutOfBlocks):
        bm.append_batch([1, 2], [40, 40])   # 3 + 3 new blocks, 4 free
    t, lens = bm.block_tables([1, 2], 4)
    assert lens.tolist() == [16, 16] and bm.num_free() == 4


def test_manager_from_several_threads(lib):
    import threading
    bm = pa.BlockManager(4096)
    errors = []

    def worker(base):
        try:
            for k in range(200):
                sid = base * 1000 + k
                bm.allocate(sid, 20)
                bm.append(sid, 30)
                bm.free(sid)
        except Exception as e:   # pragma: no cover - reported below
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors and bm.num_free() == 4096


@pytest.mark.parametrize("seed", range(25))
def test_native_prefix_caching_matches_the_oracle(lib, seed):
    rnd = random.Random(500 + seed)
    nblocks = rnd.choice([6, 20, 64])
    bm = pa.BlockManager(nblocks)
    ref = RefManager(nblocks)
    bases = [[rnd.randint(0, 3) for _ in range(rnd.randint(0, 70))] for _ in range(4)]
    toks_of = {}
    nid = 0
    for _ in range(250):
        live = sorted(ref.tables)
        op = rnd.random()
        if op < 0.45 or not live:
            toks = list(rnd.choice(bases)) + [rnd.randint(0, 3) for _ in range(rnd.randint(0, 40))]
            try:
                want = ref.allocate_cached(nid, toks)
            except RefOOM:
                with pytest.raises(pa.OutOfBlocks):
                    bm.allocate_cached(nid, toks)
            else:
                assert bm.allocate_cached(nid, toks) == want
                toks_of[nid] = toks
            nid += 1
        elif op < 0.65:
            s = rnd.choice(live)
            k = rnd.randint(1, 20)
            try:
                want = ref.append(s, k)
            except RefOOM:
                with pytest.raises(pa.OutOfBlocks):
                    bm.append(s, k)
            else:
                assert bm.append(s, k) == (want[0], want[1])
                toks_of[s] = toks_of[s] + [rnd.randint(0, 3) for _ in range(k)]
                if rnd.random() < 0.5:
                    ref.register(s, toks_of[s])
                    bm.register(s, toks_of[s])
        elif op < 0.75:
            s = rnd.choice(live)
            ref.fork(s, nid)
            bm.fork(s, nid)
            toks_of[nid] = list(toks_of[s])
            nid += 1
        else:
            s = rnd.choice(live)
            ref.free_seq(s)
            bm.free(s)
        _same_state(bm, ref)


def test_block_tables_into_caller_buffers(lib):
    # The export can fill preallocated tensors (a serving loop's pinned
    # buffers): the same tables as a fresh export, rows past n untouched.
    bm = pa.BlockManager(32)
    for s, n in ((1, 40), (2, 5), (3, 33)):
        bm.allocate(s, n)
    want_t, want_l = bm.block_tables([3, 1, 2], 4)
    tables = torch.full((5, 4), 77, dtype=torch.int32)
    lens = torch.full((5,), 77, dtype=torch.int32)
    got_t, got_l = bm.block_tables([3, 1, 2], 4, out=(tables, lens))
    assert torch.equal(got_t, want_t) and torch.equal(got_l, want_l)
    assert got_t.data_ptr() == tables.data_ptr()
    assert (tables[3:] == 77).all() and (lens[3:] == 77).all()
    with pytest.raises(ValueError):
        bm.block_tables([1], 4, out=(tables.to(torch.int64), lens))
    with pytest.raises(ValueError):
        bm.block_tables([1], 4, out=(torch.zeros((5, 3), dtype=torch.int32), lens))
    with pytest.raises(ValueError):
        bm.block_tables([1, 2, 3], 4, out=(tables[:2], lens))
