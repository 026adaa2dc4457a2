"""Host side of beam search (no GPU): the library's block manager and the
beam decoder's step plan, with the device work done by the oracle's cache
operations and paged attention on host pools. After every step, paged
attention through the planned block tables must give exactly (bit for bit,
fp64) the oracle's dense attention over each beam's own token history: the
request's prompt rows, then one row per step from the beam it descends from
("PagedAttention: the KV cache was the bottleneck all along", section
"Virtual memory for attention")."""
import numpy as np
import pytest
import torch

import oracle
import synth.beam as SB
import synth.host as H


@pytest.fixture(scope="module")
def beam_mod():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_204_gb300.beam as m
    return m


@pytest.mark.parametrize("variant", ["beam_small", "bs4_w3", "w1"])
def test_plan_gives_each_beam_its_history(beam_mod, variant):
    cfg = SB.get("beam_small")
    if variant == "bs4_w3":
        cfg = cfg.replace(block_size=4, width=3, requests=4, seed=2071)
    elif variant == "w1":
        cfg = cfg.replace(width=1, requests=2, seed=2072)
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    dec = beam_mod.BeamDecoder(torch.empty(shape, dtype=torch.float16), torch.empty(shape, dtype=torch.float16),
                               cfg.width, cfg.max_blocks_per_seq, seed=cfg.seed)
    kc, vc = H.poison(shape, cfg.dtype), H.poison(shape, cfg.dtype)
    kw = dict(num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim, block_size=cfg.block_size, dtype=cfg.dtype)
    values = SB.HostValues(cfg)
    hist_k, hist_v = [], []
    for P in SB.prompt_lengths(cfg):
        slots = dec.admit(int(P))
        pk, pv = values.prompt(int(P))
        assert oracle.reshape_and_cache(pk, pv, kc, vc, slots, **kw) == 0
        hist_k += [pk] * cfg.width
        hist_v += [pv] * cfg.width
    W, R = cfg.width, cfg.requests
    parents_of = SB.parent_stream(cfg)
    for step in range(cfg.steps):
        parents = next(parents_of)
        nk, nv, q = values.step()
        plan = dec.plan(parents)
        assert oracle.copy_blocks(kc, vc, plan.copy_pairs, **kw) == 0
        assert oracle.reshape_and_cache(nk, nv, kc, vc, plan.slots, **kw) == 0
        paged = oracle.paged_attention(q, kc, vc, plan.block_tables, plan.context_lens, scale=cfg.scale,
                                       num_heads=cfg.num_heads, **kw)
        hist_k = [np.concatenate([hist_k[r * W + int(parents[r, i])], nk[r * W + i:r * W + i + 1]])
                  for r in range(R) for i in range(W)]
        hist_v = [np.concatenate([hist_v[r * W + int(parents[r, i])], nv[r * W + i:r * W + i + 1]])
                  for r in range(R) for i in range(W)]
        seq_start = np.concatenate([[0], np.cumsum([h.shape[0] for h in hist_k])]).astype(np.int64)
        dense = oracle.dense_attention(q, np.concatenate(hist_k), np.concatenate(hist_v), seq_start,
                                       scale=cfg.scale, num_heads=cfg.num_heads, num_kv_heads=cfg.num_kv_heads,
                                       head_dim=cfg.head_dim, dtype=cfg.dtype)
        assert np.array_equal(paged, dense), f"step {step}"
        # the grouping the plan declares: each request's beams, its common prefix
        assert np.array_equal(plan.group_start, np.arange(R + 1) * W)
        for r in range(R):
            bt = plan.block_tables[r * W:(r + 1) * W]
            k = int(plan.shared_blocks[r])
            assert (bt[:, :k] == bt[0, :k]).all()
            if W > 1 and k < bt.shape[1]:
                assert not (bt[:, k] == bt[0, k]).all() or (bt[:, k] == -1).any()
    st = dec.manager.stats()
    assert st["live_seqs"] == R * W
