"""Host-side block manager used to lay out synthetic workloads.

It hands out physical blocks on demand as sequences grow, shares blocks
between forked sequences with reference counts, and records a copy-on-write
pair when a sequence is about to write into a block that another sequence
still references ("PagedAttention: the KV cache was the bottleneck all along",
section "Virtual memory for attention": blocks are acquired as a sequence
grows; sampled completions share the prompt's blocks and copy only on
divergence).

It only produces block ids, slots and (src, dst) pairs: it never touches K/V
values.
"""
from __future__ import annotations

import numpy as np


class OutOfBlocks(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        # free list in a random order: physical placement is scattered
        self._free = [int(b) for b in rng.permutation(self.num_blocks)[::-1]]
        self.ref = np.zeros(self.num_blocks, dtype=np.int32)
        self.tables: list[list[int]] = []
        self.lengths: list[int] = []
        self.cow_pairs: list[tuple[int, int]] = []

    # -- allocation ---------------------------------------------------------
    def _allocate(self) -> int:
        if not self._free:
            raise OutOfBlocks("pool exhausted")
        b = self._free.pop()
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self._free.append(b)

    @property
    def num_free(self) -> int:
        return len(self._free)

    # -- sequences ----------------------------------------------------------
    def new_seq(self) -> int:
        self.tables.append([])
        self.lengths.append(0)
        return len(self.tables) - 1

    def fork(self, seq: int) -> int:
        """A new sequence sharing every block of `seq` (reference counts +1)."""
        child = self.new_seq()
        self.tables[child] = list(self.tables[seq])
        self.lengths[child] = self.lengths[seq]
        for b in self.tables[child]:
            self.ref[b] += 1
        return child

    def free_seq(self, seq: int) -> None:
        for b in self.tables[seq]:
            self._release(b)
        self.tables[seq] = []
        self.lengths[seq] = 0

    def append_slot(self, seq: int) -> int:
        """Slot for the next token of `seq`. Allocates a block at a block
        boundary; copies a shared last block before writing into it."""
        table, pos = self.tables[seq], self.lengths[seq]
        off = pos % self.block_size
        if off == 0:
            table.append(self._allocate())
        elif self.ref[table[-1]] > 1:
            old = table[-1]
            new = self._allocate()
            self.cow_pairs.append((old, new))
            self.ref[old] -= 1
            table[-1] = new
        self.lengths[seq] = pos + 1
        return table[-1] * self.block_size + off

    def append(self, seq: int, n: int) -> list[int]:
        return [self.append_slot(seq) for _ in range(n)]

    def blocks_needed(self, seq: int) -> int:
        return -(-self.lengths[seq] // self.block_size)

    def waste_tokens(self, seq: int) -> int:
        """Unfilled slots at the end of the sequence's last block."""
        return len(self.tables[seq]) * self.block_size - self.lengths[seq]
