"""Paged prefill on the GPU against the oracle.

A system prompt is written once into a root sequence's blocks; users fork it
(sharing those blocks, copying the partly filled last one on write) and
append their own prompts; the prefill attends each user's tokens causally to
the system prompt and to their own earlier tokens ("PagedAttention: the KV
cache was the bottleneck all along", sections "What is left" and "Virtual
memory for attention"). The same writes, copies and attention run in the
oracle on host pools; outputs must agree within the tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth.prefill as SP
from gpu_helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}
DEV = torch.device("cuda", 0)


def up(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(TD[dtype])


def t64(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_prefill(cfg, lay, vals, kc_d, vc_d, err):
    import paged_kv_cache_204_gb300 as pkv
    if lay.system_slots.size:
        pkv.reshape_and_cache(up(vals.system_k, cfg.dtype), up(vals.system_v, cfg.dtype), kc_d, vc_d,
                              t64(lay.system_slots), dev_err=err)
    if lay.copy_pairs.size:
        pkv.copy_blocks(kc_d, vc_d, t64(lay.copy_pairs), dev_err=err)
    pkv.reshape_and_cache(up(vals.user_k, cfg.dtype), up(vals.user_v, cfg.dtype), kc_d, vc_d, t64(lay.user_slots),
                          dev_err=err)
    out = torch.empty((lay.total_queries, cfg.num_heads, cfg.head_dim), dtype=TD[cfg.dtype], device=DEV)
    pkv.paged_attention_prefill(out, up(vals.q, cfg.dtype), kc_d, vc_d, t64(lay.block_tables), t64(lay.context_lens),
                                t64(lay.query_start), cfg.scale, lay.max_query_len, dev_err=err)
    return out


def oracle_prefill(cfg, lay, vals, users=None):
    kc, vc = SP.host_pools(cfg)
    kw = dict(num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim, block_size=cfg.block_size, dtype=cfg.dtype)
    if lay.system_slots.size:
        oracle.reshape_and_cache(vals.system_k, vals.system_v, kc, vc, lay.system_slots, **kw)
    oracle.copy_blocks(kc, vc, lay.copy_pairs, **kw)
    oracle.reshape_and_cache(vals.user_k, vals.user_v, kc, vc, lay.user_slots, **kw)
    u = np.arange(cfg.users) if users is None else np.asarray(users)
    qs = lay.query_start
    rows = np.concatenate([np.arange(qs[i], qs[i + 1]) for i in u])
    sub_qs = np.concatenate([[0], np.cumsum(qs[u + 1] - qs[u])]).astype(np.int32)
    ref = oracle.paged_prefill(np.ascontiguousarray(vals.q[rows]), kc, vc, lay.block_tables[u], lay.context_lens[u],
                               sub_qs, scale=cfg.scale, num_heads=cfg.num_heads, threads=8, **kw)
    return ref, rows


CASES = {
    "small": {},
    "no_system_prompt": dict(system_len=0, seed=2091),
    "bs16_d128_mha": dict(block_size=16, head_dim=128, num_heads=4, num_kv_heads=4, system_len=100,
                          user_len=("uniform", 1, 200), seed=2092),
    "bf16_bs32_gqa4": dict(dtype="bf16", block_size=32, head_dim=128, num_heads=8, num_kv_heads=2, system_len=64,
                           user_len=("uniform", 60, 140), users=4, seed=2093),
    "short_users": dict(user_len=("uniform", 1, 3), users=5, system_len=16, seed=2094),
    "tile_edges": dict(user_len=("fixed", (63, 64, 65, 128, 129)), users=5, system_len=0, num_blocks=400, seed=2095),
    # users with no new tokens (n = 0) between users with some: their tiles do nothing
    "zero_query_users": dict(user_len=("fixed", (0, 70, 1, 0)), users=4, system_len=20, seed=2096),
    # head_dim 64 over long contexts: one query tile per user (every K/V tile's S issued two tiles
    # ahead), and pairs of query tiles whose second tile reads K/V tiles past the first's causal end
    "d64_long_single_tile": dict(system_len=300, user_len=("uniform", 60, 120), users=3, num_blocks=400,
                                 seed=2098),
    "d64_long_pairs": dict(system_len=200, user_len=("uniform", 130, 250), users=3, num_blocks=400, seed=2099),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    cfg = SP.get("prefill_small").replace(**CASES[name])
    lay = SP.build(cfg)
    vals = SP.host_values(cfg, lay)
    kc, vc = SP.host_pools(cfg)
    kc_d, vc_d = up(kc, cfg.dtype), up(vc, cfg.dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_prefill(cfg, lay, vals, kc_d, vc_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, rows = oracle_prefill(cfg, lay, vals)
    assert_close(to_f64(out)[rows], ref, name)


def test_prefill_full_size_sampled():
    """The benchmark's shape (16 users, a 1024-token system prompt, 40 heads):
    every query of three users against the oracle's prefill over the blocks
    those users read (copied back from the device pools after the writes)."""
    cfg = SP.get("prefill")
    lay = SP.build(cfg)
    vals = SP.host_values(cfg, lay)
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    kc_d = torch.full(shape, float("nan"), dtype=TD[cfg.dtype], device=DEV)
    vc_d = torch.full(shape, float("nan"), dtype=TD[cfg.dtype], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_prefill(cfg, lay, vals, kc_d, vc_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    u = np.array([0, 7, 15])
    bt = lay.block_tables[u]
    ids = np.unique(bt[bt >= 0])
    remap = np.full(cfg.num_blocks, -1, dtype=np.int32)
    remap[ids] = np.arange(ids.size, dtype=np.int32)
    bt_c = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(ids.astype(np.int64)).to(DEV)
    kc = kc_d[idx].cpu().view(torch.int16).numpy().view(np.uint16)
    vc = vc_d[idx].cpu().view(torch.int16).numpy().view(np.uint16)
    qs = lay.query_start
    rows = np.concatenate([np.arange(qs[i], qs[i + 1]) for i in u])
    sub_qs = np.concatenate([[0], np.cumsum(qs[u + 1] - qs[u])]).astype(np.int32)
    ref = oracle.paged_prefill(np.ascontiguousarray(vals.q[rows]), kc, vc, bt_c, lay.context_lens[u], sub_qs,
                               scale=cfg.scale, num_heads=cfg.num_heads, num_kv_heads=cfg.num_kv_heads,
                               head_dim=cfg.head_dim, block_size=cfg.block_size, dtype=cfg.dtype, threads=3)
    assert_close(to_f64(out)[rows], ref, "full-size sampled")


def test_prefill_device_errors_are_reported_and_skipped():
    """A block id out of range sets PKV_DEV_ERR_BLOCK_ID (its rows read as
    zeros, nothing faults); a sequence with more queries than tokens sets
    PKV_DEV_ERR_CONTEXT_LEN and is skipped; the context stays usable."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = SP.get("prefill_small")
    lay = SP.build(cfg)
    vals = SP.host_values(cfg, lay)
    kc, vc = SP.host_pools(cfg)
    kc_d, vc_d = up(kc, cfg.dtype), up(vc, cfg.dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_prefill(cfg, lay, vals, kc_d, vc_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bad_bt = lay.block_tables.copy()
    bad_bt[1, 0] = cfg.num_blocks + 5
    out2 = torch.empty_like(out)
    pkv.paged_attention_prefill(out2, up(vals.q, cfg.dtype), kc_d, vc_d, t64(bad_bt), t64(lay.context_lens),
                                t64(lay.query_start), cfg.scale, lay.max_query_len, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEV_ERR_BLOCK_ID
    err.zero_()
    bad_cl = lay.context_lens.copy()
    bad_cl[0] = int(lay.query_start[1] - lay.query_start[0]) - 1  # fewer tokens than queries
    pkv.paged_attention_prefill(out2, up(vals.q, cfg.dtype), kc_d, vc_d, t64(lay.block_tables), t64(bad_cl),
                                t64(lay.query_start), cfg.scale, lay.max_query_len, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEV_ERR_CONTEXT_LEN
    # the context is still fine: a normal call gives the same result as before
    err.zero_()
    out3 = torch.empty_like(out)
    pkv.paged_attention_prefill(out3, up(vals.q, cfg.dtype), kc_d, vc_d, t64(lay.block_tables),
                                t64(lay.context_lens), t64(lay.query_start), cfg.scale, lay.max_query_len,
                                dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and torch.equal(out3, out)


def _ramp_values(cfg, lay, growth, seed):
    """Keys that point more and more along one direction u as their position
    grows, and queries near u: every query's scores rise steadily along the
    context, so the running maximum keeps moving by more than the kernel's
    re-basing threshold and the tensor-memory rescale of O runs on most
    tiles."""
    import synth.host as H
    rng = np.random.default_rng(seed)
    Hkv, D = cfg.num_kv_heads, cfg.head_dim
    u = rng.standard_normal(D)
    sys_pos = np.arange(cfg.system_len, dtype=float)
    user_pos = np.concatenate([np.arange(int(lay.query_start[i + 1] - lay.query_start[i]), dtype=float)
                               + cfg.system_len for i in range(cfg.users)])
    keys = lambda pos: growth * pos[:, None, None] * u[None, None, :] + rng.standard_normal((pos.size, Hkv, D))
    nrm = lambda shape: rng.standard_normal(shape)
    st = lambda x: H.round_to_storage(x, cfg.dtype)
    n = lay.total_queries
    return SP.PrefillValues(system_k=st(keys(sys_pos)), system_v=st(nrm((cfg.system_len, Hkv, D))),
                            user_k=st(keys(user_pos)), user_v=st(nrm((n, Hkv, D))),
                            q=st(u[None, None, :] + 0.3 * nrm((n, cfg.num_heads, D))))


SCALE_CASES = {
    # scores rising ~10 (base 2) per 64-token tile: O is re-based on most tiles
    "rising_scores": dict(growth=0.01, scale=None),
    # a negative scale: the kernel scales before the maximum instead of after
    "negative_scale": dict(growth=0.0, scale=-0.125),
    # scale 0: every visible token weighs the same (the mean of the visible V rows)
    "zero_scale": dict(growth=0.0, scale=0.0),
}


@pytest.mark.parametrize("name", list(SCALE_CASES))
def test_prefill_rescale_and_scale_sign(name):
    case = SCALE_CASES[name]
    cfg = SP.get("prefill_small").replace(dtype="bf16", head_dim=128, block_size=16, num_heads=4, num_kv_heads=2,
                                          system_len=100, user_len=("uniform", 150, 300), users=3, num_blocks=300,
                                          seed=2101)
    if case["scale"] is not None:
        cfg = cfg.replace(scale=case["scale"])
    lay = SP.build(cfg)
    vals = _ramp_values(cfg, lay, case["growth"], seed=2102)
    kc, vc = SP.host_pools(cfg)
    kc_d, vc_d = up(kc, cfg.dtype), up(vc, cfg.dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_prefill(cfg, lay, vals, kc_d, vc_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, rows = oracle_prefill(cfg, lay, vals)
    assert_close(to_f64(out)[rows], ref, name)


def test_prefill_wait_timeout_is_reported_and_context_survives():
    """With a wait limit of 0 the prefill's roles (TMA loads, MMA issue,
    softmax) give up at their first wait that is not already complete: the
    call reports PKV_DEV_ERR_TIMEOUT and nothing else, and every CTA lets its
    own TMA loads land and its MMAs complete before it frees its tensor
    memory. The next call with the default limit matches the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = SP.get("prefill_small").replace(dtype="bf16", block_size=16, head_dim=128, num_heads=4,
                                          num_kv_heads=4, system_len=100, user_len=("uniform", 100, 300),
                                          seed=2097)
    lay = SP.build(cfg)
    vals = SP.host_values(cfg, lay)
    kc, vc = SP.host_pools(cfg)
    kc_d, vc_d = up(kc, cfg.dtype), up(vc, cfg.dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_prefill(cfg, lay, vals, kc_d, vc_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q, bt, cl, qs = up(vals.q, cfg.dtype), t64(lay.block_tables), t64(lay.context_lens), t64(lay.query_start)
    old = pkv.get_wait_timeout_ns()
    try:
        pkv.set_wait_timeout_ns(0)
        pkv.paged_attention_prefill(torch.empty_like(out), q, kc_d, vc_d, bt, cl, qs, cfg.scale,
                                    lay.max_query_len, dev_err=err)
        torch.cuda.synchronize()
        code = int(err.item())
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT
    assert code & ~pkv.DEV_ERR_TIMEOUT == 0
    err.zero_()
    out2 = torch.empty_like(out)
    pkv.paged_attention_prefill(out2, q, kc_d, vc_d, bt, cl, qs, cfg.scale, lay.max_query_len, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, rows = oracle_prefill(cfg, lay, vals)
    assert_close(to_f64(out2)[rows], ref, "prefill after timeout")
