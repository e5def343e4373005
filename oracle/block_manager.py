"""Plain model of the KV block manager: TEST INFRASTRUCTURE ONLY.

What the pages fix ("vLLM 部署深度指南", section 代码层面理解, the
PagedAttentionKVCache sketch; "vLLM GitHub 项目…", section 二 items 1 and 4,
section 三 item 1):
  * the free list starts as every block id in increasing order and a block is
    taken from its front;
  * a sequence of n tokens holds ceil(n / block_size) blocks; when a token
    falls past the last block a new block is taken and appended to the
    sequence's block table;
  * running out of free blocks is an out-of-memory error;
  * sequences may share physical blocks (parallel sampling / beam search share
    a prompt's blocks), and a finished sequence's blocks are released at once.
Readings where the pages are silent (each listed in the design notes):
  * a failed allocation changes nothing (the sketch would leave a partial
    table behind; all-or-nothing is the plainest usable reading);
  * released blocks go to the back of the free list, in table order, when no
    other table still references them (reference counting);
  * writing a token into a block that another table also references first
    moves the writer to a private copy (copy-on-write): a new block is taken,
    the copy (old -> new) is recorded for the cache, the old block loses one
    reference.

Prefix caching ("vLLM 部署深度指南", Prefix Caching 加速 table and the
PagedAttention table's 前缀共享 row; "vLLM高性能推理引擎实战解密", section 3.1
PagedAttention内存管理机制, cross-request sharing: requests with the same
prefix share its KV cache)
is read as: a full block can serve any request whose tokens, from the first
up to that block's last, are the same.  A cached block is found by the key
(parent block, the parent's generation, the block's tokens) -- exact, no
hashing shortcuts -- where the generation counts how often a block id has
been handed out, so a key naming a block that was since reused never
matches.  Released cached blocks stay findable until the allocator hands
them out again (then their key is dropped).  At least one prompt token is
always left to compute, so a fully cached prompt recomputes its last block.

Everything is plain Python lists and dicts, step by step.
"""

from collections import deque


class OutOfBlocks(Exception):
    """The pool has too few free blocks for the request (the pages' OOMError)."""


class BlockManager:
    def __init__(self, num_blocks, block_size=16):
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free = deque(range(num_blocks))
        self.ref = [0] * num_blocks
        self.tables = {}   # seq_id -> list of physical block ids
        self.lens = {}     # seq_id -> tokens held
        self.gen = [0] * num_blocks   # times each block id was handed out
        self.cache = {}    # (parent block, parent gen, tokens) -> cached block
        self.key_of = {}   # cached block -> its key

    def blocks_for(self, num_tokens):
        return (num_tokens + self.block_size - 1) // self.block_size

    def num_free(self):
        return len(self.free)

    def _take(self):
        b = self.free.popleft()
        if b in self.key_of:               # handing out a cached block evicts it
            del self.cache[self.key_of.pop(b)]
        self.gen[b] += 1
        self.ref[b] = 1
        return b

    def _drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def allocate(self, seq_id, num_tokens):
        """A new sequence holding ``num_tokens`` tokens."""
        assert seq_id not in self.tables and num_tokens >= 0
        need = self.blocks_for(num_tokens)
        if need > len(self.free):
            raise OutOfBlocks(f"need {need} blocks, {len(self.free)} free")
        self.tables[seq_id] = [self._take() for _ in range(need)]
        self.lens[seq_id] = num_tokens

    def append(self, seq_id, n):
        """Reserve ``n`` new tokens at the end of ``seq_id``.

        Returns ``(slots, copies)``: the slot (block * block_size + offset) of
        each new token, and the (src, dst) block copies the cache must perform
        before those slots are written (copy-on-write of a shared last block).
        """
        table = self.tables[seq_id]
        L = self.lens[seq_id]
        bs = self.block_size
        cow = n > 0 and L % bs != 0 and self.ref[table[L // bs]] > 1
        new_blocks = self.blocks_for(L + n) - len(table)
        if new_blocks + (1 if cow else 0) > len(self.free):
            raise OutOfBlocks(f"need {new_blocks + int(cow)} blocks, {len(self.free)} free")
        copies = []
        if cow:
            old = table[L // bs]
            new = self._take()
            copies.append((old, new))
            self.ref[old] -= 1          # still referenced by another table
            table[L // bs] = new
        for _ in range(new_blocks):
            table.append(self._take())
        slots = []
        for pos in range(L, L + n):
            slots.append(table[pos // bs] * bs + pos % bs)
        self.lens[seq_id] = L + n
        return slots, copies

    def fork(self, parent, child):
        """``child`` shares every block of ``parent`` (same tokens so far)."""
        assert child not in self.tables
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, seq_id):
        """Release a finished sequence's blocks (those no other table holds)."""
        for b in self.tables.pop(seq_id):
            self._drop(b)
        del self.lens[seq_id]

    def block_table(self, seq_id, width):
        t = self.tables[seq_id]
        return t + [-1] * (width - len(t))

    # ---------------------------------------------------------- prefix caching

    def _key(self, parent, tokens):
        return (parent, self.gen[parent] if parent >= 0 else 0, tuple(tokens))

    def register(self, seq_id, tokens):
        """Make the full blocks of ``seq_id`` findable; ``tokens`` are its token
        ids from the first (at least its length's worth of full blocks)."""
        bs = self.block_size
        table = self.tables[seq_id]
        parent = -1
        for j in range(min(len(tokens), self.lens[seq_id]) // bs):
            b = table[j]
            key = self._key(parent, tokens[j * bs:(j + 1) * bs])
            if key not in self.cache and b not in self.key_of:
                self.cache[key] = b
                self.key_of[b] = key
            parent = b

    def allocate_cached(self, seq_id, tokens):
        """A new sequence for the prompt ``tokens`` that reuses the longest run
        of cached full blocks from its start.  Returns the number of tokens
        whose K/V are already cached (a multiple of block_size, < len(tokens)
        unless the prompt is empty); the caller computes the rest."""
        assert seq_id not in self.tables
        bs = self.block_size
        n = len(tokens)
        reusable = (n - 1) // bs if n > 0 else 0
        hits = []
        parent = -1
        for j in range(reusable):
            b = self.cache.get(self._key(parent, tokens[j * bs:(j + 1) * bs]))
            if b is None:
                break
            hits.append(b)
            parent = b
        need = self.blocks_for(n) - len(hits)
        idle = sum(1 for b in hits if self.ref[b] == 0)   # cached blocks on the free list
        if need > len(self.free) - idle:
            raise OutOfBlocks(f"need {need} blocks, {len(self.free) - idle} free")
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
        self.tables[seq_id] = hits + [self._take() for _ in range(need)]
        self.lens[seq_id] = n
        self.register(seq_id, tokens)
        return len(hits) * bs
