"""Plain-Python block manager and block copy, the oracle of the library's manager.

TEST INFRASTRUCTURE ONLY (see ``oracle.py``).  Written from the definition:
the KV cache is a pool of fixed-size physical blocks placed anywhere; each
sequence's block table lists, in order, the physical blocks holding its
tokens, and only the blocks needed are allocated ("PagedAttention, décodage
spéculatif, MoE et Blackwell", §1, pagination de type système d'exploitation;
"LLM inference optimization: KV cache", §4.1, §4.2).  Sequences forked from one
another share physical blocks; a shared block is copied before it is written
(copy on write; same §1, partage de mémoire; §4.2).

Readings (the pages give no policy): a new block is the lowest-numbered free
block; a block is shared while more than one sequence lists it; a write needs
a copy only when it goes into a shared block that already holds tokens (a
fresh block is never shared).
"""
from __future__ import annotations

import numpy as np


class OutOfBlocks(Exception):
    pass


class BlockManager:
    def __init__(self, num_blocks, block_size):
        self.block_size = block_size
        self.refs = [0] * num_blocks
        self.tables = {}          # seq id -> list of physical block ids
        self.tokens = {}          # seq id -> number of tokens

    def free_blocks(self):
        return [b for b, r in enumerate(self.refs) if r == 0]

    def _new_block(self):
        free = self.free_blocks()
        if not free:
            raise OutOfBlocks()
        b = min(free)
        self.refs[b] = 1
        return b

    def add_sequence(self, seq, n):
        if seq in self.tables or n < 0:
            raise ValueError(seq)
        need = -(-n // self.block_size)
        if need > len(self.free_blocks()):
            raise OutOfBlocks()
        self.tables[seq] = [self._new_block() for _ in range(need)]
        self.tokens[seq] = n

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables or parent == child:
            raise ValueError((parent, child))
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            self.refs[b] += 1

    def append_slot(self, seq):
        """Slot of the sequence's next token, and the (src, dst) copy it needs (or None)."""
        if seq not in self.tables:
            raise ValueError(seq)
        table = self.tables[seq]
        pos = self.tokens[seq]
        offset = pos % self.block_size
        copy = None
        if offset == 0:
            table.append(self._new_block())
        elif self.refs[table[-1]] > 1:
            old = table[-1]
            new = self._new_block()
            self.refs[old] -= 1
            table[-1] = new
            copy = (old, new)
        self.tokens[seq] = pos + 1
        return table[-1] * self.block_size + offset, copy

    def free_sequence(self, seq):
        if seq not in self.tables:
            raise ValueError(seq)
        for b in self.tables.pop(seq):
            self.refs[b] -= 1
        del self.tokens[seq]


def copy_blocks(k_cache, v_cache, pairs):
    """New (k, v) pools with block dst replaced by block src for every pair."""
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    for src, dst in pairs:
        k[dst] = k_cache[src]
        v[dst] = v_cache[src]
    return k, v
