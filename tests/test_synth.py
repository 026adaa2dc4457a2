"""Seeded input generators and the host block manager (no GPU)."""
import json
import os

import numpy as np
import pytest

import synth
import synth.host as H
from synth.blockmgr import BlockManager

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("name", sorted(synth.PRESETS))
def test_structure_invariants(name):
    cfg = synth.get(name)
    st = synth.build(cfg)
    bs = cfg.block_size
    assert st.num_seqs == cfg.num_seqs
    lo, hi = cfg.lengths[-2], cfg.lengths[-1]
    if cfg.tail is not None:
        lo, hi = lo + cfg.tail[1], hi + cfg.tail[2]
    assert st.context_lens.min() >= lo and st.context_lens.max() <= hi
    assert st.max_context_len == st.context_lens.max() <= cfg.max_blocks_per_seq * bs
    nblk = -(-st.context_lens // bs)
    for s in range(st.num_seqs):
        row = st.block_tables[s]
        assert (row[:nblk[s]] >= 0).all() and (row[nblk[s]:] == synth.PAD_BLOCK).all()
        assert row[:nblk[s]].max() < cfg.num_blocks
    # waste: only the unfilled tail of the last block
    assert (st.waste_tokens >= 0).all() and (st.waste_tokens < bs).all()
    assert np.array_equal(st.waste_tokens, nblk * bs - st.context_lens)
    # each physical block belongs to one sequence unless shared by forks
    ids, counts = np.unique(st.block_tables[st.block_tables >= 0], return_counts=True)
    if cfg.samples == 1:
        assert counts.max() == 1
    else:
        assert counts.max() <= cfg.samples
        assert np.array_equal(st.refcount[ids], counts)
    # new rows: one per sequence at its last position (new-token configs)
    if cfg.new_token:
        last = st.context_lens - 1
        expect = st.block_tables[np.arange(st.num_seqs), last // bs].astype(np.int64) * bs + last % bs
        assert np.array_equal(st.slot_mapping, expect)
    assert np.array_equal(st.prefix_lens + np.diff(st.new_start), st.context_lens)


def test_copy_on_write_reading():
    """Per prompt whose length is not a multiple of block_size, the first
    samples to write into the shared partial block copy it; the last writes
    in place. Full prompt blocks stay shared by every sample."""
    cfg = synth.get("cow")
    st = synth.build(cfg)
    bs, S = cfg.block_size, cfg.samples
    partial = (st.prefix_lens[::S] % bs) != 0
    assert st.copy_pairs.shape[0] == (S - 1) * int(partial.sum())
    for p in range(cfg.num_seqs // S):
        rows = st.block_tables[p * S:(p + 1) * S]
        full = st.prefix_lens[p * S] // bs
        assert (rows[:, :full] == rows[0, :full]).all()          # shared full blocks
        if partial[p]:
            last = rows[:, full]
            assert len(set(last.tolist())) == S                    # diverged
            src = st.copy_pairs[np.isin(st.copy_pairs[:, 1], last)][:, 0]
            assert (src == rows[-1, full]).all()                   # copies of the in-place writer's block


def test_block_manager_fork_free():
    mgr = BlockManager(16, 4, np.random.default_rng(0))
    a = mgr.new_seq()
    mgr.append(a, 6)                   # 2 blocks
    b = mgr.fork(a)
    assert mgr.num_free == 14 and mgr.ref[mgr.tables[a]].tolist() == [2, 2]
    mgr.append(b, 1)                   # writes into shared partial block -> copy
    assert len(mgr.cow_pairs) == 1 and mgr.tables[a][1] != mgr.tables[b][1]
    mgr.append(a, 1)                   # now private -> in place
    assert len(mgr.cow_pairs) == 1
    mgr.free_seq(b)
    mgr.free_seq(a)
    assert mgr.num_free == 16 and (mgr.ref == 0).all()


def test_seeded_determinism():
    cfg = synth.get("llama7b")
    a = H.generate(cfg, num_seqs=3)
    b = H.generate(cfg, num_seqs=3)
    for x, y in ((a.q, b.q), (a.prefill_k, b.prefill_k), (a.prefill_v, b.prefill_v)):
        assert np.array_equal(x, y)
    assert np.array_equal(a.st.block_tables, b.st.block_tables)
    c = H.generate(cfg, seed=cfg.seed + 1, num_seqs=3)
    assert not np.array_equal(a.q, c.q)


@pytest.mark.parametrize("name", ["tiny", "llama13b", "cow"])
def test_poison_rows(name):
    cfg = synth.get(name)
    hw = H.generate(cfg, num_seqs=6 if cfg.samples > 1 else 4)
    rows = np.arange(cfg.block_size)
    empty = rows[None, :] >= hw.st.prefill_rows[:, None]
    pk = H.is_poison(hw.prefill_k)                      # [U, Hkv, bs, D]
    assert np.array_equal(pk, np.broadcast_to(empty[:, None, :, None], pk.shape))
    assert np.array_equal(H.is_poison(hw.prefill_v), pk)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40, 3.0e38])
    got = H.round_to_storage(x, "bf16")
    back = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == -2.5


def test_golden_kv_size_per_sequence():
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_llama13b_sequence.json")))
    cfg = synth.get("llama13b")
    assert cfg.kv_bytes_per_token() == 20480
    total = cfg.kv_bytes_per_token() * g["model_shape_not_on_the_pages"]["layers"] * \
        g["model_shape_not_on_the_pages"]["max_tokens"]
    assert abs(total / 1e9 - g["value_gb"]) <= g["printed_precision_gb"]


def test_golden_waste_bound():
    g = json.load(open(os.path.join(GOLDEN, "paged_waste_bound.json")))
    for name in g["applies_to"]:
        st = synth.build(synth.get(name))
        allocated = (-(-st.context_lens // st.cfg.block_size) * st.cfg.block_size).sum()
        assert st.waste_tokens.sum() / allocated < g["max_waste_fraction"], name
