"""Beam search over the paged KV cache on the GPU, step after step.

Each step the library's block manager forks and ends beams and reserves the
new rows' slots; the kernels copy shared partly filled blocks, write the new
rows and run the grouped decode with one group per request. After every step
each beam's output must equal the oracle's dense attention over that beam's
own token history: its request's prompt rows, then the row written at each
step by the beam it descends from ("PagedAttention: the KV cache was the
bottleneck all along", section "Virtual memory for attention": beams share
prefixes, are forked and discarded, and copy a block only when they
diverge). This checks the copies, the writes, the tables and the grouping
end to end without trusting the block manager."""
import numpy as np
import pytest
import torch

import oracle
import synth.beam as SB
from synth.device import fill_poison
from gpu_helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def up(a: np.ndarray, dtype: str, dev) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a if dtype == "f32" else a.view(np.int16))
    return t.to(dev).view(TD[dtype])


def dense_reference(cfg, hist_k, hist_v, q):
    """Oracle: softmax attention of each beam's query over its own history."""
    seq_start = np.concatenate([[0], np.cumsum([h.shape[0] for h in hist_k])]).astype(np.int64)
    k = np.ascontiguousarray(np.concatenate(hist_k))
    v = np.ascontiguousarray(np.concatenate(hist_v))
    return oracle.dense_attention(q, k, v, seq_start, scale=cfg.scale, num_heads=cfg.num_heads,
                                  num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim, dtype=cfg.dtype)


@pytest.mark.parametrize("variant", ["beam_small", "beam_small_bs16_mha", "beam_small_bf16_w2"])
def test_beam_steps_match_dense_history(variant):
    import paged_kv_cache_204_gb300 as pkv
    from paged_kv_cache_204_gb300.beam import BeamDecoder

    cfg = SB.get("beam_small")
    if variant == "beam_small_bs16_mha":
        cfg = cfg.replace(block_size=16, num_heads=4, num_kv_heads=4, head_dim=128, seed=2061)
    elif variant == "beam_small_bf16_w2":
        cfg = cfg.replace(dtype="bf16", width=2, requests=5, seed=2062)
    dev = torch.device("cuda", 0)
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    kc = torch.empty(shape, dtype=TD[cfg.dtype], device=dev)
    vc = torch.empty(shape, dtype=TD[cfg.dtype], device=dev)
    fill_poison(kc)
    fill_poison(vc)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dec = BeamDecoder(kc, vc, cfg.width, cfg.max_blocks_per_seq, seed=cfg.seed)
    values = SB.HostValues(cfg)
    hist_k, hist_v = [], []  # per batch row: the beam's token rows so far
    for P in SB.prompt_lengths(cfg):
        pk, pv = values.prompt(int(P))
        dec.add_request(up(pk, cfg.dtype, dev), up(pv, cfg.dtype, dev), dev_err=err)
        hist_k += [pk] * cfg.width
        hist_v += [pv] * cfg.width
    W, R = cfg.width, cfg.requests
    parents_of = SB.parent_stream(cfg)
    copies = 0
    for step in range(cfg.steps):
        parents = next(parents_of)
        nk, nv, q = values.step()
        plan = dec.plan(parents)
        copies += plan.copy_pairs.shape[0]
        dp = dec.upload(plan)
        out = dec.run(dp, up(nk, cfg.dtype, dev), up(nv, cfg.dtype, dev), up(q, cfg.dtype, dev), cfg.scale,
                      torch.empty(q.shape, dtype=TD[cfg.dtype], device=dev), dev_err=err)
        plain = torch.empty_like(out)
        ws = pkv.new_workspace(R * W, cfg.num_heads, cfg.head_dim, dp.max_context_len, device=dev)
        pkv.paged_attention_decode(plain, up(q, cfg.dtype, dev), kc, vc, dp.block_tables, dp.context_lens, cfg.scale,
                                   dp.max_context_len, workspace=ws, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error word {int(err.item()):#x} at step {step}"
        # histories of the new beams: the parent's rows, then the row just written
        new_k, new_v = [], []
        for r in range(R):
            for i in range(W):
                row = r * W + i
                par = r * W + int(parents[r, i])
                new_k.append(np.concatenate([hist_k[par], nk[row:row + 1]]))
                new_v.append(np.concatenate([hist_v[par], nv[row:row + 1]]))
        hist_k, hist_v = new_k, new_v
        assert np.array_equal(plan.context_lens, [h.shape[0] for h in hist_k])
        ref = dense_reference(cfg, hist_k, hist_v, q)
        assert_close(to_f64(out), ref, f"{variant} grouped, step {step}")
        assert_close(to_f64(plain), ref, f"{variant} plain, step {step}")
        # every request's beams were declared as sharing at least what they share
        for r in range(R):
            assert plan.shared_blocks[r] == dec.manager.common_prefix(dec.requests[r])
    assert copies > 0  # the steps did exercise copy-on-write
