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

    def blocks_for(self, num_tokens):
        return (num_tokens + self.block_size - 1) // self.block_size

    def num_free(self):
        return len(self.free)

    def _take(self):
        b = self.free.popleft()
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
