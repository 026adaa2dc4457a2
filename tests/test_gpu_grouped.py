"""Grouped decode (siblings reading shared prefix blocks once) through the C
ABI: same results as the oracle (and as plain decode) on copy-on-write
batches, including groups of one, more than four members, empty tails, a
zero-length prompt, grouped-query heads, block sizes 8/16/32, a wrong
grouping promise and an invalid grouping (both flagged and still correct)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as SD
import synth.host as H
from gpu_helpers import assert_close, device_error, to_f64

pytestmark = pytest.mark.gpu


def _run_grouped(dw, group_start, shared_blocks, err, ws=None):
    import paged_kv_cache_204_gb300 as pkv
    st, cfg = dw.st, dw.cfg
    if dw.copy_pairs.numel():
        pkv.copy_blocks(dw.k_cache, dw.v_cache, dw.copy_pairs, dev_err=err)
    if dw.slot_mapping.numel():
        pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=err)
    gs = torch.as_tensor(np.asarray(group_start, np.int32), device="cuda")
    sb = torch.as_tensor(np.asarray(shared_blocks, np.int32), device="cuda")
    if ws is None:
        ws = pkv.new_grouped_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim, st.max_context_len,
                                       sb.numel())
    out = torch.full_like(dw.q, float("nan"))
    pkv.paged_attention_decode_grouped(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                       dw.context_lens, cfg.scale, st.max_context_len, gs, sb, ws,
                                       dev_err=err)
    return out


def _check(st, cfg, **kw):
    hw = H.generate(cfg, st=st)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_grouped(dw, st.group_start if "gs" not in kw else kw["gs"],
                       st.shared_blocks if "sb" not in kw else kw["sb"], err)
    code = device_error(err)
    ref, _, _ = oracle.decode_step(hp, hw, threads=8)
    assert_close(to_f64(out), ref, cfg.name)
    return code


@pytest.mark.parametrize("name,B", [("cow", 12), ("cow", 96)])
def test_copy_on_write_workload(name, B):
    cfg = synth.get(name)
    st = synth.build(cfg, num_seqs=B)
    assert (st.shared_blocks > 0).all()
    assert _check(st, cfg) == 0


SHAPES = [(40, [0, 5, 20]), (100, [3]), (64, [0, 0]), (200, [1, 2, 3, 4, 5, 6]), (0, [7, 9]),
          (333, [17, 1]), (16, [0, 1, 2, 3, 4])]


@pytest.mark.parametrize("dtype,D,bs,Hkv,G", [("f16", 128, 16, 4, 1), ("bf16", 64, 8, 2, 2),
                                               ("f32", 128, 32, 2, 1), ("bf16", 128, 16, 2, 4),
                                               ("f16", 64, 32, 3, 3)])
def test_group_shapes(dtype, D, bs, Hkv, G):
    cfg = synth.get("cow").replace(num_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                   dtype=dtype, num_blocks=3000, lengths=("fixed", (400,)),
                                   tail=("fixed", (64,)), scale=1.0 / np.sqrt(D))
    st = synth.build_grouped(cfg, SHAPES)
    assert _check(st, cfg) == 0


@pytest.mark.parametrize("groups", [128, 129, 150])
def test_many_groups(groups):
    """More groups than the grouping check's blocks hold warps (8 per block):
    the check still covers every group, the result is the oracle's, and a
    wrong shared-blocks promise in one group among many is flagged."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("cow").replace(samples=2, num_heads=4, num_kv_heads=4, num_blocks=6000,
                                   lengths=("uniform", 16, 160), tail=("uniform", 1, 40))
    st = synth.build(cfg, num_seqs=2 * groups)
    assert len(st.shared_blocks) == groups
    assert _check(st, cfg) == 0
    lie = st.shared_blocks.copy()
    lie[groups // 2] += 2                              # one group promises blocks that differ
    assert _check(st, cfg, sb=lie) == pkv.DEV_ERR_GROUP


def test_wrong_shared_blocks_promise_is_flagged_and_still_correct():
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("cow").replace(num_heads=4, num_kv_heads=4, num_blocks=3000,
                                   lengths=("fixed", (400,)), tail=("fixed", (64,)))
    st = synth.build_grouped(cfg, SHAPES)
    lie = st.shared_blocks + 3                         # promises blocks that differ
    code = _check(st, cfg, sb=lie)
    assert code == pkv.DEV_ERR_GROUP


def test_invalid_grouping_is_flagged_and_ignored():
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("cow").replace(num_heads=4, num_kv_heads=4, num_blocks=3000,
                                   lengths=("fixed", (400,)), tail=("fixed", (64,)))
    st = synth.build_grouped(cfg, SHAPES)
    bad = st.group_start.copy()
    bad[-1] -= 1                                       # does not cover the last sequence
    code = _check(st, cfg, gs=bad)
    assert code == pkv.DEV_ERR_GROUP


def test_workspace_reuse_and_plain_agreement():
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("cow").replace(num_heads=8, num_kv_heads=8, num_blocks=4000)
    st = synth.build(cfg, num_seqs=24)
    hw = H.generate(cfg, st=st)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pkv.new_grouped_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim, st.max_context_len,
                                   len(st.shared_blocks))
    outs = [to_f64(_run_grouped(dw, st.group_start, st.shared_blocks, err, ws=ws)) for _ in range(3)]
    assert device_error(err) == 0
    plain = torch.empty_like(dw.q)
    pkv.paged_attention_decode(plain, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                               cfg.scale, st.max_context_len,
                               workspace=pkv.new_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim,
                                                           st.max_context_len))
    for o in outs:
        assert_close(o, to_f64(plain), "grouped vs plain")


def test_wait_timeout_is_reported_and_context_survives():
    """With a wait limit of 0 the grouped kernel's warps give up at their
    first wait that is not already complete: they report PKV_DEV_ERR_TIMEOUT
    (and nothing else), let their own copies land and return. After the
    workspace is cleared, the next call with the default limit matches the
    oracle."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("cow").replace(num_heads=8, num_kv_heads=8, num_blocks=4000)
    st = synth.build(cfg, num_seqs=24)
    hw = H.generate(cfg, st=st)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pkv.new_grouped_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim, st.max_context_len,
                                   len(st.shared_blocks))
    old = pkv.get_wait_timeout_ns()
    try:
        pkv.set_wait_timeout_ns(0)
        _run_grouped(dw, st.group_start, st.shared_blocks, err, ws=ws)
        code = device_error(err)
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT
    assert code & ~pkv.DEV_ERR_TIMEOUT == 0
    # the cache writes ran before the timed-out attention: restart from fresh pools
    dw = SD.from_host(hw)
    err.zero_()
    ws.zero_()  # a call that reported a device error may leave piece counters set
    out = _run_grouped(dw, st.group_start, st.shared_blocks, err, ws=ws)
    assert device_error(err) == 0
    ref, _, _ = oracle.decode_step(hp, hw, threads=8)
    assert_close(to_f64(out), ref, "grouped after timeout")
