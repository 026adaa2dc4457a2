"""Reference model of the paged KV block manager — TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this module; the product never does.

What it models ("PagedAttention: the KV cache was the bottleneck all along",
section "Virtual memory for attention"): a sequence's tokens sit in
fixed-size blocks reached through its block table; a sequence takes a new
block only when a token starts one; samples (or beams) forked from a
sequence share its blocks; a sequence that writes into a block another live
sequence still uses gets its own copy first (copy-on-write).

It does not allocate physical blocks. Each logical block of each sequence
refers to a block *identity* (a plain integer that stands for "these token
rows"); two sequences share physical memory exactly when they refer to the
same identity. So every quantity the pages talk about — blocks in use,
copies, filled slots, shared blocks — follows from the identities alone,
and any allocator that is correct must agree with it on all of them, while
its physical block ids are free to differ (any one-to-one relabelling).

Plain Python, slow on purpose: state is recomputed from the tables.
"""
from __future__ import annotations

import copy


class OutOfBlocks(RuntimeError):
    pass


class BlockModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = int(num_blocks)
        self.bs = int(block_size)
        self.tables: dict[int, list[int]] = {}  # handle -> identities of its logical blocks
        self.lengths: dict[int, int] = {}
        self._next_handle = 0
        self._next_identity = 0
        self.copies = 0

    # -- derived state (recomputed every time) -----------------------------
    def holders(self, ident: int) -> int:
        """Live sequences whose tables refer to the identity."""
        return sum(1 for t in self.tables.values() if ident in t)

    def used_identities(self) -> set[int]:
        return {i for t in self.tables.values() for i in t}

    def used_blocks(self) -> int:
        return len(self.used_identities())

    def free_blocks(self) -> int:
        return self.num_blocks - self.used_blocks()

    def shared_blocks(self) -> int:
        return sum(1 for i in self.used_identities() if self.holders(i) > 1)

    def filled_slots(self) -> int:
        """Slots of the blocks in use that hold a token of some live sequence:
        for each identity, the furthest token any holder keeps in it."""
        reach: dict[int, int] = {}
        for h, t in self.tables.items():
            for j, ident in enumerate(t):
                kept = min(self.bs, self.lengths[h] - j * self.bs)
                reach[ident] = max(reach.get(ident, 0), kept)
        return sum(reach.values())

    def logical_blocks(self) -> int:
        """Blocks the live sequences would hold with private copies."""
        return sum(len(t) for t in self.tables.values())

    def logical_tokens(self) -> int:
        return sum(self.lengths.values())

    def stats(self) -> dict:
        return {"num_blocks": self.num_blocks, "free_blocks": self.free_blocks(),
                "used_blocks": self.used_blocks(), "shared_blocks": self.shared_blocks(),
                "filled_slots": self.filled_slots(), "logical_blocks": self.logical_blocks(),
                "logical_tokens": self.logical_tokens(), "live_seqs": len(self.tables),
                "cow_copies": self.copies}

    # -- operations ----------------------------------------------------------
    def _new_identity(self) -> int:
        self._next_identity += 1
        return self._next_identity

    def add_seq(self) -> int:
        h = self._next_handle
        self._next_handle += 1
        self.tables[h] = []
        self.lengths[h] = 0
        return h

    def fork(self, parent: int) -> int:
        h = self.add_seq()
        self.tables[h] = list(self.tables[parent])
        self.lengths[h] = self.lengths[parent]
        return h

    def free_seq(self, h: int) -> None:
        del self.tables[h]
        del self.lengths[h]

    def blocks_needed(self, h: int, n: int) -> tuple[int, bool]:
        """(new identities an append of n tokens takes, whether it copies)."""
        if n == 0:
            return 0, False
        L = self.lengths[h]
        copies = L % self.bs != 0 and self.holders(self.tables[h][-1]) > 1
        starts = sum(1 for t in range(L, L + n) if t % self.bs == 0)
        return starts + (1 if copies else 0), copies

    def append(self, h: int, n: int) -> bool:
        """Append n tokens one at a time; True when the first one copied a
        shared block. Raises OutOfBlocks (nothing changed) when the pool is
        too small."""
        need, copies = self.blocks_needed(h, n)
        if need > self.free_blocks():
            raise OutOfBlocks(f"need {need}, free {self.free_blocks()}")
        copied = False
        for _ in range(n):
            L = self.lengths[h]
            if L % self.bs == 0:
                self.tables[h].append(self._new_identity())
            elif self.holders(self.tables[h][-1]) > 1:
                self.tables[h][-1] = self._new_identity()  # private copy of the shared rows
                self.copies += 1
                copied = True
            self.lengths[h] = L + 1
        assert copied == copies
        return copied

    def beam_step(self, beams, parents, n_new: int = 1) -> list[int]:
        """New beam i continues beams[parents[i]]: the parent's first new beam
        keeps its sequence, later ones fork it; beams no new beam continues
        end; then each new beam appends n_new tokens in order. Raises
        OutOfBlocks with nothing changed when the step does not fit."""
        trial = copy.deepcopy(self)
        for j, b in enumerate(beams):
            if j not in parents:
                trial.free_seq(b)
        new, kept = [], set()
        for j in parents:
            if j in kept:
                new.append(trial.fork(beams[j]))
            else:
                kept.add(j)
                new.append(beams[j])
        for h in new:
            trial.append(h, n_new)
        self.__dict__.update(trial.__dict__)
        return new

    def beam_step_many(self, rows, parent_rows, n_new: int = 1) -> list[list[int]]:
        """The same step for several requests at once, in three passes over
        all of them: every beam that no new beam of its own request continues
        ends; then every new beam takes its sequence (first child keeps the
        parent's, later ones fork it); then every new beam appends n_new
        tokens, request by request and in order within a request. Raises
        OutOfBlocks with nothing changed when the whole step does not fit."""
        trial = copy.deepcopy(self)
        for beams, parents in zip(rows, parent_rows):
            for j, b in enumerate(beams):
                if j not in parents:
                    trial.free_seq(b)
        out = []
        for beams, parents in zip(rows, parent_rows):
            new, kept = [], set()
            for j in parents:
                if j in kept:
                    new.append(trial.fork(beams[j]))
                else:
                    kept.add(j)
                    new.append(beams[j])
            out.append(new)
        for new in out:
            for h in new:
                trial.append(h, n_new)
        self.__dict__.update(trial.__dict__)
        return out

    def common_prefix(self, handles) -> int:
        ts = [self.tables[h] for h in handles]
        k = 0
        while all(k < len(t) for t in ts) and all(t[k] == ts[0][k] for t in ts):
            k += 1
        return k
