"""Seeded structure of a decode step: context lengths, block tables, the blocks
that already hold K/V before the step, and the step's writes (slots of new
rows, copy-on-write pairs). No K/V values here (see host.py / device.py).

Lengths:
  ("fixed", (l0, l1, ...))              the given lengths, repeated cyclically
  ("uniform", lo, hi)                   integers uniform in [lo, hi]
  ("lognormal", median, sigma, lo, hi)  rint(exp(ln(median) + sigma * z)), clipped
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .blockmgr import BlockManager
from .configs import DecodeConfig

PAD_BLOCK = -1  # block table entries past a sequence's last block


@dataclass
class Structure:
    cfg: DecodeConfig
    context_lens: np.ndarray     # int32 [B]: tokens attention reads (after the step's writes)
    block_tables: np.ndarray     # int32 [B, max_blocks_per_seq], PAD_BLOCK past the end
    max_context_len: int
    prefill_blocks: np.ndarray   # int64 [U]: blocks holding K/V before the step
    prefill_rows: np.ndarray     # int32 [U]: rows of each such block already written
    copy_pairs: np.ndarray       # int64 [n, 2]: step's copy-on-write (src, dst)
    slot_mapping: np.ndarray     # int64 [T]: step's new K/V rows
    refcount: np.ndarray         # int32 [num_blocks] after the step
    waste_tokens: np.ndarray     # int32 [B]: unfilled slots of each sequence's last block
    prefix_lens: np.ndarray      # int32 [B]: tokens already cached before the step
    prefix_tables: np.ndarray    # int32 [B, MB]: block tables before the step (shared rows for forks)
    new_start: np.ndarray        # int64 [B+1]: slot_mapping rows [new_start[s], new_start[s+1]) are s's
    group_start: np.ndarray | None = None    # int32 [G+1]: forks of one prompt are consecutive sequences
    shared_blocks: np.ndarray | None = None  # int32 [G]: leading blocks every member maps identically

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    def used_blocks(self) -> np.ndarray:
        """Every physical block referenced by the step, sorted."""
        bt = self.block_tables[self.block_tables >= 0]
        parts = [bt.astype(np.int64), self.prefill_blocks, self.copy_pairs.reshape(-1),
                 self.slot_mapping // self.cfg.block_size]
        return np.unique(np.concatenate([p.astype(np.int64) for p in parts]))

    def unique_kv_tokens(self) -> int:
        """Distinct (block, row) cache slots attention reads, all sequences.
        Shared prompt rows count once."""
        bs = self.cfg.block_size
        seen = {}
        for s in range(self.num_seqs):
            L = int(self.context_lens[s])
            for j in range(-(-L // bs)):
                b = int(self.block_tables[s, j])
                rows = min(bs, L - j * bs)
                seen[b] = max(seen.get(b, 0), rows)
        return int(sum(seen.values()))


def draw_lengths(spec: tuple, n: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        _, lo, hi = spec
        return rng.integers(lo, hi + 1, size=n).astype(np.int64)
    if kind == "lognormal":
        _, median, sigma, lo, hi = spec
        z = rng.standard_normal(n)
        return np.clip(np.rint(np.exp(np.log(median) + sigma * z)), lo, hi).astype(np.int64)
    if kind == "fixed":
        vals = np.asarray(spec[1], dtype=np.int64)
        return np.resize(vals, n)
    raise ValueError(f"unknown length distribution {spec!r}")


def build(cfg: DecodeConfig, seed: int | None = None, num_seqs: int | None = None) -> Structure:
    """Lay out one decode step of `cfg`. `num_seqs` overrides the batch
    (prompts * samples for copy-on-write configs must stay a multiple)."""
    seed = cfg.seed if seed is None else seed
    B = cfg.num_seqs if num_seqs is None else num_seqs
    len_rng = np.random.default_rng([seed, 1])
    mgr = BlockManager(cfg.num_blocks, cfg.block_size, np.random.default_rng([seed, 2]))
    prefill_rows: dict[int, int] = {}

    def prefill(seq: int, n: int) -> None:
        for slot in mgr.append(seq, n):
            b = slot // cfg.block_size
            prefill_rows[b] = prefill_rows.get(b, 0) + 1

    slots: list[int] = []
    new_count: dict[int, int] = {}
    snapshot: dict[int, tuple[int, list[int]]] = {}
    if cfg.samples > 1:
        if B % cfg.samples:
            raise ValueError("num_seqs must be a multiple of samples")
        prompts = B // cfg.samples
        plen = draw_lengths(cfg.lengths, prompts, len_rng)
        tails = draw_lengths(cfg.tail, B, len_rng)
        seqs = []
        for p in range(prompts):
            root = mgr.new_seq()
            prefill(root, int(plen[p]))
            seqs.append([root] + [mgr.fork(root) for _ in range(cfg.samples - 1)])
        order = [s for group in seqs for s in group]
        group_sizes = [len(gr) for gr in seqs]
        for s in order:
            snapshot[s] = (mgr.lengths[s], list(mgr.tables[s]))
        for i, s in enumerate(order):  # divergence: each sample appends its own tail
            slots.extend(mgr.append(s, int(tails[i])))
            new_count[s] = int(tails[i])
    else:
        group_sizes = None
        lens = draw_lengths(cfg.lengths, B, len_rng)
        order = []
        for i in range(B):
            s = mgr.new_seq()
            n_new = 1 if cfg.new_token else 0
            prefill(s, int(lens[i]) - n_new)
            order.append(s)
            snapshot[s] = (mgr.lengths[s], list(mgr.tables[s]))
        if cfg.new_token:
            for s in order:
                slots.append(mgr.append_slot(s))
                new_count[s] = 1

    MB = cfg.max_blocks_per_seq
    bt = np.full((B, MB), PAD_BLOCK, dtype=np.int32)
    cl = np.zeros(B, dtype=np.int32)
    waste = np.zeros(B, dtype=np.int32)
    pbt = np.full((B, MB), PAD_BLOCK, dtype=np.int32)
    plen = np.zeros(B, dtype=np.int32)
    nstart = np.zeros(B + 1, dtype=np.int64)
    for row, s in enumerate(order):
        t = mgr.tables[s]
        bt[row, :len(t)] = t
        cl[row] = mgr.lengths[s]
        waste[row] = mgr.waste_tokens(s)
        plen[row], pt = snapshot[s]
        pbt[row, :len(pt)] = pt
        nstart[row + 1] = nstart[row] + new_count.get(s, 0)
    pb = np.array(sorted(prefill_rows), dtype=np.int64)
    pr = np.array([prefill_rows[b] for b in pb], dtype=np.int32)
    gstart, shared = _groups(bt, group_sizes)
    return Structure(cfg=cfg, context_lens=cl, block_tables=bt,
                     max_context_len=int(cl.max()) if B else 0,
                     prefill_blocks=pb, prefill_rows=pr,
                     copy_pairs=np.array(mgr.cow_pairs, dtype=np.int64).reshape(-1, 2),
                     slot_mapping=np.array(slots, dtype=np.int64),
                     refcount=mgr.ref.copy(), waste_tokens=waste, prefix_lens=plen,
                     prefix_tables=pbt, new_start=nstart, group_start=gstart, shared_blocks=shared)


def _groups(bt: np.ndarray, group_sizes):
    """Group boundaries and the number of leading block-table entries every
    member of a group shares (read off the final tables)."""
    if group_sizes is None:
        return None, None
    gstart = np.concatenate([[0], np.cumsum(group_sizes)]).astype(np.int32)
    shared = np.zeros(len(group_sizes), dtype=np.int32)
    for g in range(len(group_sizes)):
        rows = bt[gstart[g]:gstart[g + 1]]
        same = (rows == rows[0]).all(axis=0) & (rows[0] >= 0)
        shared[g] = int(np.argmin(same)) if not same.all() else same.size
    return gstart, shared


def build_grouped(cfg: DecodeConfig, prompts: list, seed: int | None = None) -> Structure:
    """A copy-on-write batch with explicit shapes: prompts = [(prompt_len,
    [tail_len, ...]), ...]; each prompt is prefilled, forked into one sequence
    per tail, and each fork appends its tail (tails may be 0). Sequences of one
    prompt are consecutive and form a group."""
    seed = cfg.seed if seed is None else seed
    mgr = BlockManager(cfg.num_blocks, cfg.block_size, np.random.default_rng([seed, 2]))
    prefill_rows: dict[int, int] = {}
    order, group_sizes, snapshot, new_count, slots = [], [], {}, {}, []
    for plen, tails in prompts:
        root = mgr.new_seq()
        for slot in mgr.append(root, int(plen)):
            b = slot // cfg.block_size
            prefill_rows[b] = prefill_rows.get(b, 0) + 1
        members = [root] + [mgr.fork(root) for _ in range(len(tails) - 1)]
        order += members
        group_sizes.append(len(members))
        for m in members:
            snapshot[m] = (mgr.lengths[m], list(mgr.tables[m]))
    i = 0
    for plen, tails in prompts:
        for tl in tails:
            s = order[i]
            slots.extend(mgr.append(s, int(tl)))
            new_count[s] = int(tl)
            i += 1
    B, MB = len(order), cfg.max_blocks_per_seq
    bt = np.full((B, MB), PAD_BLOCK, dtype=np.int32)
    pbt = np.full((B, MB), PAD_BLOCK, dtype=np.int32)
    cl = np.zeros(B, dtype=np.int32)
    plen_a = np.zeros(B, dtype=np.int32)
    waste = np.zeros(B, dtype=np.int32)
    nstart = np.zeros(B + 1, dtype=np.int64)
    for row, s in enumerate(order):
        t = mgr.tables[s]
        bt[row, :len(t)] = t
        cl[row] = mgr.lengths[s]
        waste[row] = mgr.waste_tokens(s)
        plen_a[row], pt = snapshot[s]
        pbt[row, :len(pt)] = pt
        nstart[row + 1] = nstart[row] + new_count.get(s, 0)
    pb = np.array(sorted(prefill_rows), dtype=np.int64)
    pr = np.array([prefill_rows[b] for b in pb], dtype=np.int32)
    gstart, shared = _groups(bt, group_sizes)
    return Structure(cfg=cfg, context_lens=cl, block_tables=bt, max_context_len=int(cl.max()),
                     prefill_blocks=pb, prefill_rows=pr,
                     copy_pairs=np.array(mgr.cow_pairs, dtype=np.int64).reshape(-1, 2),
                     slot_mapping=np.array(slots, dtype=np.int64), refcount=mgr.ref.copy(),
                     waste_tokens=waste, prefix_lens=plen_a, prefix_tables=pbt, new_start=nstart,
                     group_start=gstart, shared_blocks=shared)
