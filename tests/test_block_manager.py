"""Host block manager (no GPU needed).

1. The oracle's block model is pinned to things other than itself: closed
   forms for one sequence and for a prompt forked into samples, a brute-force
   count of distinct block contents from token labels, and planted mistakes
   that those pins catch.
2. The library's manager (include/pkv_block_manager.h) agrees with the model
   after every operation of seeded random operation sequences: every counter
   equal, physical ids a one-to-one relabelling of the model's block
   identities, slots and copy-on-write pairs consistent with the tables.
3. The memory figures the pages give ("PagedAttention: the KV cache was the
   bottleneck all along", sections "Virtual memory for attention" and "The
   number that made us read the code"), measured on the synthetic workloads.
"""
import copy
import json
import os

import numpy as np
import pytest

import synth
from oracle.block_model import BlockModel, OutOfBlocks as ModelOutOfBlocks
from synth.replay import replay

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def pb():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_204_gb300.block_manager as m
    return m


def ceil_div(a, b):
    return -(-a // b)


# ---- 1. pins of the model ------------------------------------------------------

@pytest.mark.parametrize("bs", [1, 8, 16])
def test_model_single_sequence_closed_form(bs):
    for L in [0, 1, bs - 1, bs, bs + 1, 5 * bs + 3, 100]:
        m = BlockModel(1000, bs)
        s = m.add_seq()
        m.append(s, L)
        st = m.stats()
        assert st["used_blocks"] == ceil_div(L, bs) == st["logical_blocks"]
        assert st["filled_slots"] == L and st["logical_tokens"] == L
        assert st["cow_copies"] == 0 and st["shared_blocks"] == 0
        assert st["used_blocks"] * bs - L < bs  # only the last block's tail is empty


def fork_closed_form(P, tails, bs):
    """Blocks, copies, shared blocks and filled slots after a prompt of P
    tokens is forked into len(tails) samples that each append tails[i] >= 1
    tokens: full prompt blocks stay shared; a partial prompt block is copied
    by every sample but the last to write, so each sample ends up with its own
    partial block holding the P % bs prompt rows plus its tail."""
    k, full, part = len(tails), P // bs, P % bs
    used = full + sum(ceil_div(part + t, bs) for t in tails)
    copies = k - 1 if part else 0
    filled = full * bs + k * part + sum(tails)
    return used, copies, (full if k > 1 else 0), filled


@pytest.mark.parametrize("bs", [4, 16])
def test_model_fork_closed_form(bs):
    rng = np.random.default_rng(5)
    for _ in range(40):
        P = int(rng.integers(1, 6 * bs))
        tails = [int(t) for t in rng.integers(1, 3 * bs, size=int(rng.integers(1, 5)))]
        m = BlockModel(10000, bs)
        root = m.add_seq()
        m.append(root, P)
        seqs = [root] + [m.fork(root) for _ in range(len(tails) - 1)]
        for s, t in zip(seqs, tails):
            m.append(s, t)
        used, copies, shared, filled = fork_closed_form(P, tails, bs)
        st = m.stats()
        assert (st["used_blocks"], st["cow_copies"], st["shared_blocks"], st["filled_slots"]) == \
            (used, copies, shared, filled), (P, tails)
        assert st["logical_blocks"] == sum(ceil_div(P + t, bs) for t in tails)


def random_ops(seed, n_ops, bs, num_blocks, max_append=20):
    """A seeded operation list over sequence *positions* (indices into the
    list of live sequences at the time of the operation)."""
    rng = np.random.default_rng(seed)
    ops = []
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.15:
            ops.append(("add",))
        elif r < 0.35:
            ops.append(("fork", int(rng.integers(1 << 30))))
        elif r < 0.45:
            ops.append(("free", int(rng.integers(1 << 30))))
        elif r < 0.55:
            ops.append(("batch", int(rng.integers(1 << 30)), int(rng.integers(1, 6)), int(rng.integers(1, 4))))
        else:
            ops.append(("append", int(rng.integers(1 << 30)), int(rng.integers(0, max_append))))
    return ops


def distinct_views(labels: dict, bs: int) -> tuple[int, int]:
    """Brute force from content alone: each appended token carries a unique
    label and a fork copies its parent's label list. Memory must hold every
    distinct block content (the labels in one block of one sequence); shared
    physical blocks are exactly the equal contents. Returns (blocks, slots)."""
    views = set()
    for lab in labels.values():
        for j in range(0, len(lab), bs):
            views.add(tuple(lab[j:j + bs]))
    return len(views), sum(len(v) for v in views)


def run_model_with_labels(model_cls, seed, bs=4, num_blocks=64, n_ops=150):
    m = model_cls(num_blocks, bs)
    labels, live, nxt = {}, [], [0]

    def add_tokens(h, n):
        labels[h] += list(range(nxt[0], nxt[0] + n))
        nxt[0] += n

    for op in random_ops(seed, n_ops, bs, num_blocks):
        try:
            if op[0] == "add" or not live:
                h = m.add_seq()
                labels[h] = []
                live.append(h)
            elif op[0] == "fork":
                p = live[op[1] % len(live)]
                h = m.fork(p)
                labels[h] = list(labels[p])
                live.append(h)
            elif op[0] == "free":
                h = live.pop(op[1] % len(live))
                m.free_seq(h)
                del labels[h]
            else:
                h = live[op[1] % len(live)]
                n = op[2] if op[0] == "append" else op[3]
                m.append(h, n)
                add_tokens(h, n)
        except ModelOutOfBlocks:
            pass
        yield m, labels


def test_model_matches_brute_force_views():
    for seed in range(12):
        for m, labels in run_model_with_labels(BlockModel, seed):
            assert (m.used_blocks(), m.filled_slots()) == distinct_views(labels, m.bs)


# planted mistakes in the model: each must fail one of the pins above
class NoCopyModel(BlockModel):
    """Writes into a shared block instead of copying it."""
    def append(self, h, n):
        need = sum(1 for t in range(self.lengths[h], self.lengths[h] + n) if t % self.bs == 0)
        if need > self.free_blocks():
            raise ModelOutOfBlocks("")
        for _ in range(n):
            if self.lengths[h] % self.bs == 0:
                self.tables[h].append(self._new_identity())
            self.lengths[h] += 1
        return False


class AlwaysCopyModel(BlockModel):
    """Copies a partial last block even when it holds it alone."""
    def append(self, h, n):
        if n and self.lengths[h] % self.bs:
            self.tables[h][-1] = self._new_identity()
            self.copies += 1
        for _ in range(n):
            if self.lengths[h] % self.bs == 0:
                self.tables[h].append(self._new_identity())
            self.lengths[h] += 1
        return False


class DeepForkModel(BlockModel):
    """A fork copies every block instead of sharing."""
    def fork(self, parent):
        h = self.add_seq()
        self.tables[h] = [self._new_identity() for _ in self.tables[parent]]
        self.lengths[h] = self.lengths[parent]
        return h


class LateBlockModel(BlockModel):
    """Starts a new block one token late (off by one at block boundaries)."""
    def append(self, h, n):
        for _ in range(n):
            L = self.lengths[h]
            if L == 0 or (L > 1 and L % self.bs == 1):
                self.tables[h].append(self._new_identity())
            self.lengths[h] = L + 1
        return False


def _pins_pass(model_cls) -> bool:
    try:
        for bs in (4, 16):
            m = model_cls(1000, bs)
            s = m.add_seq()
            m.append(s, 5 * bs + 3)
            if m.used_blocks() != ceil_div(5 * bs + 3, bs):
                return False
            m = model_cls(10000, bs)
            root = m.add_seq()
            m.append(root, bs + 3)
            seqs = [root, m.fork(root), m.fork(root)]
            for s in seqs:
                m.append(s, 2)
            used, copies, shared, filled = fork_closed_form(bs + 3, [2, 2, 2], bs)
            st = m.stats()
            if (st["used_blocks"], st["cow_copies"], st["shared_blocks"], st["filled_slots"]) != \
                    (used, copies, shared, filled):
                return False
        for seed in range(6):
            for mm, labels in run_model_with_labels(model_cls, seed):
                if (mm.used_blocks(), mm.filled_slots()) != distinct_views(labels, mm.bs):
                    return False
    except Exception:
        return False
    return True


@pytest.mark.parametrize("mutant", [NoCopyModel, AlwaysCopyModel, DeepForkModel, LateBlockModel])
def test_model_pins_catch_planted_mistakes(mutant):
    assert _pins_pass(BlockModel)
    assert not _pins_pass(mutant)


# ---- 2. the library's manager against the model -------------------------------

def check_relabelling(prod, model, handle_of):
    """Physical ids are a one-to-one relabelling of the model's identities."""
    to_phys, to_ident = {}, {}
    for pid, h in handle_of.items():
        n, nb = prod.seq_info(pid)
        assert n == model.lengths[h] and nb == len(model.tables[h])
        bt, cl = prod.export([pid], max(nb, 1))
        assert cl[0] == n
        for j, ident in enumerate(model.tables[h]):
            phys = int(bt[0, j])
            assert 0 <= phys < model.num_blocks
            assert to_phys.setdefault(ident, phys) == phys
            assert to_ident.setdefault(phys, ident) == ident
        assert (bt[0, nb:] == -1).all()


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("bs,num_blocks", [(4, 48), (16, 300)])
def test_manager_matches_model(pb, seed, bs, num_blocks):
    prod = pb.BlockManager(num_blocks, bs, seed=seed + 1)
    model = BlockModel(num_blocks, bs)
    handle_of = {}          # product id -> model handle
    live = []               # product ids in creation order
    for op in random_ops(100 + seed, 250, bs, num_blocks, max_append=3 * bs):
        if op[0] == "add" or not live:
            pid, h = prod.add_seq(), model.add_seq()
            assert pid not in handle_of
            handle_of[pid] = h
            live.append(pid)
        elif op[0] == "fork":
            p = live[op[1] % len(live)]
            pid, h = prod.fork(p), model.fork(handle_of[p])
            handle_of[pid] = h
            live.append(pid)
        elif op[0] == "free":
            pid = live.pop(op[1] % len(live))
            prod.free_seq(pid)
            model.free_seq(handle_of.pop(pid))
        elif op[0] == "append":
            pid = live[op[1] % len(live)]
            h, n = handle_of[pid], op[2]
            n0, nb0 = prod.seq_info(pid)
            last = int(prod.export([pid], max(nb0, 1))[0][0, nb0 - 1]) if nb0 else None
            try:
                copied = model.append(h, n)
            except ModelOutOfBlocks:
                with pytest.raises(pb.OutOfBlocks):
                    prod.append(pid, n)
                assert prod.seq_info(pid) == (n0, nb0)
            else:
                slots, pair = prod.append(pid, n)
                assert (pair is not None) == copied
                bt, _ = prod.export([pid], max(prod.seq_info(pid)[1], 1))
                t = np.arange(n0, n0 + n)
                assert np.array_equal(slots, bt[0, t // bs].astype(np.int64) * bs + t % bs)
                if pair is not None:
                    assert pair[0] == last and pair[1] == bt[0, nb0 - 1] and pair[0] != pair[1]
        else:  # batch of distinct sequences
            k = min(op[2], len(live))
            start = op[1] % len(live)
            pids = [live[(start + i) % len(live)] for i in range(k)]
            counts = [op[3]] * k
            trial = copy.deepcopy(model)
            try:
                ncopies = sum(trial.append(handle_of[p], c) for p, c in zip(pids, counts))
            except ModelOutOfBlocks:
                with pytest.raises(pb.OutOfBlocks):
                    prod.append_batch(pids, counts)
            else:
                model = trial
                slots, pairs = prod.append_batch(pids, counts)
                assert len(slots) == sum(counts) and len(pairs) == ncopies
        assert prod.stats() == model.stats(), op
        check_relabelling(prod, model, handle_of)
        if len(live) >= 2:
            pick = live[:3]
            assert prod.common_prefix(pick) == model.common_prefix([handle_of[p] for p in pick])


def test_manager_placement_and_host_checks(pb):
    m = pb.BlockManager(8, 4, seed=0)
    s = m.add_seq()
    slots, _ = m.append(s, 9)
    assert list(slots) == list(range(9))                       # seed 0: ascending ids
    a, b = pb.BlockManager(50, 4, seed=9), pb.BlockManager(50, 4, seed=9)
    sa, sb = a.add_seq(), b.add_seq()
    assert np.array_equal(a.append(sa, 40)[0], b.append(sb, 40)[0])  # a seed fixes the placement
    m.free_seq(s)
    s2 = m.add_seq()
    assert s2 == s                                                # ids are reused
    assert m.append(s2, 1)[0][0] // 4 == 2                        # last freed block is handed out first
    with pytest.raises(pb.PkvError):
        m.free_seq(s2 + 5)
    with pytest.raises(pb.PkvError):
        m.append(s2, -1)
    with pytest.raises(pb.PkvError):
        m.append_batch([s2, s2], [1, 1])
    with pytest.raises(pb.PkvError):
        m.export([s2], 0)
    with pytest.raises(pb.OutOfBlocks):
        m.append(s2, 1000)
    assert m.seq_info(s2) == (1, 1)
    with pytest.raises(pb.PkvError):
        pb.BlockManager(0, 16)


def test_batch_last_sibling_writes_in_place(pb):
    """Three samples share a partial block: a batch step copies it for the
    first two and lets the last write in place, using exactly 2 new blocks."""
    m = pb.BlockManager(6, 4, seed=0)
    root = m.add_seq()
    m.append(root, 6)                        # blocks 0 (full), 1 (2 rows)
    kids = [root, m.fork(root), m.fork(root)]
    assert m.stats()["free_blocks"] == 4
    slots, pairs = m.append_batch(kids, [1, 1, 1])
    assert len(pairs) == 2 and all(p[0] == 1 for p in pairs)
    assert m.stats()["free_blocks"] == 2 and slots[2] == 1 * 4 + 2


# ---- 3. memory figures on the workloads ------------------------------------------

def manager_metrics(pb, cfg):
    m = pb.BlockManager(cfg.num_blocks, cfg.block_size, seed=cfg.seed)
    replay(m, cfg)
    st = m.stats()
    return st, pb.memory_metrics(st, cfg.block_size)


def test_waste_under_four_percent(pb):
    g = json.load(open(os.path.join(GOLDEN, "paged_waste_bound.json")))
    for name in g["applies_to"]:
        cfg = synth.get(name)
        st, mm = manager_metrics(pb, cfg)
        assert mm["waste_fraction"] < g["max_waste_fraction"], name


def test_sharing_saving_on_copy_on_write_workload(pb):
    g = json.load(open(os.path.join(GOLDEN, "paged_sharing_saving.json")))
    for name in g["applies_to"]:
        cfg = synth.get(name)
        st, mm = manager_metrics(pb, cfg)
        assert 0.3 < mm["sharing_saving"] <= g["max_sharing_saving"], (name, mm)
        # the same state as the inputs' own layout: blocks in use and copies
        s = synth.build(cfg)
        used = {int(b) for row, L in zip(s.block_tables, s.context_lens) for b in row[:ceil_div(int(L), cfg.block_size)]}
        assert st["used_blocks"] == len(used) and st["cow_copies"] == s.copy_pairs.shape[0]
        assert st["filled_slots"] == s.unique_kv_tokens()


def test_sharing_saving_matches_model_small(pb):
    cfg = synth.get("cow").replace(num_seqs=12)
    st, mm = manager_metrics(pb, cfg)
    model = BlockModel(cfg.num_blocks, cfg.block_size)
    replay(model, cfg, num_seqs=12)
    assert st == model.stats()


def test_contiguous_reservation_waste(pb):
    g = json.load(open(os.path.join(GOLDEN, "contiguous_reservation_waste.json")))
    for name in g["applies_to"]:
        cfg = synth.get(name)
        assert cfg.max_len == g["reserved_tokens_per_sequence"]
        st, mm = manager_metrics(pb, cfg)
        reserved = st["live_seqs"] * cfg.max_len
        contiguous = 1.0 - st["logical_tokens"] / reserved
        assert g["min_waste_fraction"] <= contiguous <= g["max_waste_fraction"], (name, contiguous)
        assert mm["waste_fraction"] < contiguous / 10


# ---- beam search steps ---------------------------------------------------------------

def draw_parents(rng, W):
    """Skewed parent choice: better-ranked beams are continued more often,
    so some beams end and others continue more than once."""
    p = np.arange(W, 0, -1, dtype=float) ** 2
    return [int(x) for x in rng.choice(W, size=W, p=p / p.sum())]


def test_model_beam_step_matches_brute_force_views():
    rng = np.random.default_rng(11)
    for bs in (2, 4):
        m = BlockModel(100000, bs)
        labels, nxt = {}, 0
        reqs = []
        for r in range(3):
            root = m.add_seq()
            P = int(rng.integers(1, 5 * bs))
            m.append(root, P)
            labels[root] = list(range(nxt, nxt + P))
            nxt += P
            W = 4
            beams = [root] + [m.fork(root) for _ in range(W - 1)]
            for b in beams[1:]:
                labels[b] = list(labels[root])
            reqs.append(beams)
        for step in range(12):
            for r, beams in enumerate(reqs):
                parents = draw_parents(rng, len(beams))
                old = {b: list(labels[b]) for b in beams}
                new = m.beam_step(beams, parents, 1)
                for b in beams:
                    labels.pop(b, None)
                for i, h in enumerate(new):
                    labels[h] = old[beams[parents[i]]] + [nxt]
                    nxt += 1
                reqs[r] = new
            assert (m.used_blocks(), m.filled_slots()) == distinct_views(labels, bs)
            assert m.logical_tokens() == sum(len(v) for v in labels.values())


class KeepDeadBeamsModel(BlockModel):
    """Planted mistake: beams nobody continues are not ended."""
    def beam_step(self, beams, parents, n_new=1):
        new, kept = [], set()
        for j in parents:
            new.append(self.fork(beams[j]) if j in kept else beams[j])
            kept.add(j)
        for h in new:
            self.append(h, n_new)
        return new


def test_beam_pin_catches_kept_dead_beams():
    rng = np.random.default_rng(3)
    m = KeepDeadBeamsModel(100000, 4)
    root = m.add_seq()
    m.append(root, 10)
    beams = [root] + [m.fork(root) for _ in range(3)]
    labels = {b: list(range(10)) for b in beams}
    nxt = 10
    for _ in range(6):
        parents = [0, 0, 1, 1]
        old = {b: list(labels[b]) for b in beams}
        new = m.beam_step(beams, parents)
        labels = {h: old[beams[parents[i]]] + [nxt + i] for i, h in enumerate(new)}
        nxt += 4
        beams = new
    assert (m.used_blocks(), m.filled_slots()) != distinct_views(labels, 4)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bs,num_blocks", [(4, 60), (16, 2000)])
def test_manager_beam_steps_match_model(pb, seed, bs, num_blocks):
    rng = np.random.default_rng(200 + seed)
    prod = pb.BlockManager(num_blocks, bs, seed=seed + 3)
    model = BlockModel(num_blocks, bs)
    handle_of = {}
    reqs = []
    for r in range(3):
        P = int(rng.integers(1, 4 * bs))
        pr, mr = prod.add_seq(), model.add_seq()
        handle_of[pr] = mr
        try:
            model.append(mr, P)
            prod.append(pr, P)
        except ModelOutOfBlocks:
            with pytest.raises(pb.OutOfBlocks):
                prod.append(pr, P)
            continue
        beams = [pr]
        for _ in range(int(rng.integers(2, 6)) - 1):
            c = prod.fork(pr)
            handle_of[c] = model.fork(mr)
            beams.append(c)
        reqs.append(beams)
    for step in range(30):
        for r, beams in enumerate(reqs):
            parents = draw_parents(rng, len(beams))
            n_new = int(rng.integers(1, 3))
            try:
                mnew = model.beam_step([handle_of[b] for b in beams], parents, n_new)
            except ModelOutOfBlocks:
                with pytest.raises(pb.OutOfBlocks):
                    prod.beam_step(beams, parents, n_new)
                continue
            new, slots, pairs = prod.beam_step(beams, parents, n_new)
            assert len(slots) == len(new) * n_new
            gone = [b for j, b in enumerate(beams) if j not in parents]
            for b in gone:
                handle_of.pop(b)
            for pid, h in zip(new, mnew):
                handle_of[pid] = h
            reqs[r] = list(new)
            assert len(pairs) <= len(new)
        assert prod.stats() == model.stats(), step
        check_relabelling(prod, model, handle_of)
        for beams in reqs:
            assert prod.common_prefix(beams) == model.common_prefix([handle_of[b] for b in beams])


def test_beam_step_host_checks(pb):
    m = pb.BlockManager(20, 4)
    a = m.add_seq()
    m.append(a, 5)
    b = m.fork(a)
    with pytest.raises(pb.PkvError):
        m.beam_step([a, b], [0, 2])
    with pytest.raises(pb.PkvError):
        m.beam_step([a, a], [0, 1])
    with pytest.raises(pb.OutOfBlocks):
        m.beam_step([a, b], [0, 0], 100)
    assert m.stats()["live_seqs"] == 2 and m.seq_info(a) == (5, 2) and m.seq_info(b) == (5, 2)


# ---- batched beam steps (all requests of a decode step in one call) ---------------------

def beam_requests(rng, m, bs, n_req, share_prompt):
    """Requests of 2-5 beams each. With share_prompt every request's root is a
    fork of one common prompt, so blocks are shared across requests too."""
    labels, reqs, nxt = {}, [], 0
    common = None
    if share_prompt:
        common = m.add_seq()
        P = int(rng.integers(1, 4 * bs))
        m.append(common, P)
        labels[common] = list(range(P))
        nxt = P
    for r in range(n_req):
        if common is not None:
            root = m.fork(common)
            labels[root] = list(labels[common])
        else:
            root = m.add_seq()
            labels[root] = []
        P = int(rng.integers(1, 3 * bs))
        m.append(root, P)
        labels[root] += list(range(nxt, nxt + P))
        nxt += P
        beams = [root]
        for _ in range(int(rng.integers(2, 6)) - 1):
            c = m.fork(root)
            labels[c] = list(labels[root])
            beams.append(c)
        reqs.append(beams)
    return labels, reqs, nxt, common


@pytest.mark.parametrize("share_prompt", [False, True])
def test_model_beam_step_many_matches_brute_force_views(share_prompt):
    rng = np.random.default_rng(12 + share_prompt)
    for bs in (2, 4):
        m = BlockModel(100000, bs)
        labels, reqs, nxt, _ = beam_requests(rng, m, bs, 4, share_prompt)
        for step in range(10):
            parents = [draw_parents(rng, len(b)) for b in reqs]
            old = {b: list(labels[b]) for beams in reqs for b in beams}
            new = m.beam_step_many(reqs, parents, 2)
            for beams in reqs:
                for b in beams:
                    labels.pop(b, None)
            for beams, ps, nb in zip(reqs, parents, new):
                for i, h in enumerate(nb):
                    labels[h] = old[beams[ps[i]]] + [nxt, nxt + 1]
                    nxt += 2
            reqs = new
            assert (m.used_blocks(), m.filled_slots()) == distinct_views(labels, bs)
            assert m.logical_tokens() == sum(len(v) for v in labels.values())


def test_model_beam_step_many_is_per_request_steps_without_sharing():
    """Requests that share no block: the batched step leaves the same
    counters and tables (up to block identity) as one step per request."""
    rng = np.random.default_rng(21)
    a = BlockModel(100000, 4)
    _, reqs, _, _ = beam_requests(rng, a, 4, 3, False)
    b = copy.deepcopy(a)
    for step in range(8):
        parents = [draw_parents(rng, len(x)) for x in reqs]
        new_a = a.beam_step_many(reqs, parents, 1)
        new_b = [b.beam_step(x, p, 1) for x, p in zip(reqs, parents)]
        assert new_a == new_b and a.stats() == b.stats()
        for row in new_a:
            assert [a.lengths[h] for h in row] == [b.lengths[h] for h in row]
            assert [a.tables[h] for h in row] == [b.tables[h] for h in row]
        reqs = new_a


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("bs,num_blocks,share", [(4, 70, False), (4, 90, True), (16, 2000, True)])
def test_manager_beam_step_many_matches_model(pb, seed, bs, num_blocks, share):
    rng = np.random.default_rng(300 + seed)
    prod = pb.BlockManager(num_blocks, bs, seed=seed + 7)
    model = BlockModel(num_blocks, bs)
    # build the same requests on both sides through the single-sequence calls
    mrng = np.random.default_rng(400 + seed)
    _, mreqs, _, mcommon = beam_requests(mrng, model, bs, 4, share)
    handle_of = {}
    prng = np.random.default_rng(400 + seed)
    preqs = []
    pcommon = None
    if share:
        pcommon = prod.add_seq()
        prod.append(pcommon, int(prng.integers(1, 4 * bs)))
        handle_of[pcommon] = mcommon
    for mbeams in mreqs:
        if pcommon is not None:
            root = prod.fork(pcommon)
        else:
            root = prod.add_seq()
        prod.append(root, int(prng.integers(1, 3 * bs)))
        beams = [root]
        for _ in range(int(prng.integers(2, 6)) - 1):
            beams.append(prod.fork(root))
        assert len(beams) == len(mbeams)
        handle_of.update(zip(beams, mbeams))
        preqs.append(beams)
    assert prod.stats() == model.stats()
    # one call per beam width (a call takes requests of equal width)
    by_width = {}
    for r, b in enumerate(preqs):
        by_width.setdefault(len(b), []).append(r)
    refused = 0
    for step in range(40):
        n_new = int(rng.integers(1, 4))
        for width, rows in sorted(by_width.items()):
            parents = [draw_parents(rng, width) for _ in rows]
            try:
                mnew = model.beam_step_many([[handle_of[b] for b in preqs[r]] for r in rows], parents, n_new)
            except ModelOutOfBlocks:
                before = prod.stats()
                with pytest.raises(pb.OutOfBlocks):
                    prod.beam_step_many([preqs[r] for r in rows], parents, n_new)
                assert prod.stats() == before
                refused += 1
                continue
            new, slots, pairs, shared = prod.beam_step_many([preqs[r] for r in rows], parents, n_new)
            assert new.shape == (len(rows), width) and len(slots) == new.size * n_new
            assert len(np.unique(slots)) == len(slots) and len(pairs) <= new.size
            for k, r in enumerate(rows):  # ended ids may be reused by any request's forks
                for j, b in enumerate(preqs[r]):
                    if j not in parents[k]:
                        handle_of.pop(b)
            for k, r in enumerate(rows):
                for pid, h in zip(new[k], mnew[k]):
                    handle_of[int(pid)] = h
                preqs[r] = [int(x) for x in new[k]]
                assert shared[k] == model.common_prefix(mnew[k])
            assert prod.stats() == model.stats(), step
            check_relabelling(prod, model, handle_of)
    if num_blocks < 100:
        assert refused > 0  # the tight pools did run out at some step


def test_beam_step_many_host_checks(pb):
    m = pb.BlockManager(30, 4)
    a = m.add_seq()
    m.append(a, 5)
    b, c, d = m.fork(a), m.fork(a), m.fork(a)
    before = m.stats()
    with pytest.raises(pb.PkvError):
        m.beam_step_many([[a, b], [c, d]], [[0, 2], [0, 0]])  # parent out of range
    with pytest.raises(pb.PkvError):
        m.beam_step_many([[a, b], [c, a]], [[0, 1], [0, 1]])  # a beam in two requests
    with pytest.raises(pb.PkvError):
        m.beam_step_many([[a, b]], [[0, 1]], -1)
    with pytest.raises(pb.OutOfBlocks):
        m.beam_step_many([[a, b], [c, d]], [[0, 0], [1, 1]], 100)
    assert m.stats() == before
    new, slots, pairs, shared = m.beam_step_many(np.zeros((0, 2), dtype=np.int32), np.zeros((0, 2), dtype=np.int32))
    assert new.shape == (0, 2) and slots.size == 0 and pairs.shape == (0, 2) and shared.size == 0
    assert m.stats() == before
    # a step that fits only because the other request's ended beams return their blocks
    m2 = pb.BlockManager(6, 4)
    x = m2.add_seq()
    m2.append(x, 8)                      # 2 full blocks
    y = m2.add_seq()
    m2.append(y, 8)                      # 2 more; 2 free
    x2, y2 = m2.fork(x), m2.fork(y)
    # request 0 keeps x only (x2 ends, its blocks stay shared with x); request 1
    # continues y twice and ends y2; 4 tokens each = 3 new blocks... needs 3 > 2 free
    with pytest.raises(pb.OutOfBlocks):
        m2.beam_step_many([[x, x2], [y, y2]], [[0, 1], [0, 0]], 4)
    assert m2.stats()["free_blocks"] == 2
    m2.free_seq(x2)
    m2.free_seq(x)                       # 2 blocks return: 4 free
    new, slots, pairs, shared = m2.beam_step_many([[y, y2]], [[0, 0]], 4)
    assert new[0, 0] == y and len(set(new[0].tolist())) == 2 and shared[0] == 2
    assert m2.stats()["free_blocks"] == 2
