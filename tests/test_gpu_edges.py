"""Edge cases of the GPU path through the C ABI: every dtype / head_dim /
block_size / grouped-head combination, context lengths at the tile and
block boundaries (including 0 and 1), segments split across many warps,
an oversized max_context_len, workspace reuse, and the device error word."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as SD
import synth.host as H
from gpu_helpers import assert_close, device_error, run_step, to_f64

pytestmark = pytest.mark.gpu

EDGE_LENS = (0, 1, 2, 15, 16, 17, 31, 33, 255, 256, 257, 511, 512, 513, 1000, 2047)

COMBOS = [  # dtype, head_dim, block_size, num_kv_heads, group
    ("f32", 64, 16, 2, 1), ("f32", 128, 8, 2, 2), ("f32", 128, 32, 1, 4),
    ("f16", 64, 8, 2, 1), ("f16", 128, 16, 2, 3), ("f16", 64, 32, 1, 8),
    ("bf16", 128, 16, 2, 1), ("bf16", 64, 16, 2, 4), ("bf16", 128, 8, 1, 2),
    ("bf16", 128, 32, 2, 5), ("f16", 128, 32, 4, 1), ("bf16", 64, 8, 3, 6),
]


def _cfg(dtype, D, bs, Hkv, G, lens=EDGE_LENS, new_token=False, nb=4000):
    return synth.DecodeConfig(
        name=f"edge_{dtype}_{D}_{bs}_{Hkv}x{G}", num_seqs=len(lens), num_heads=Hkv * G,
        num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dtype, num_blocks=nb,
        lengths=("fixed", tuple(lens)), value_scale=1.0, scale=1.0 / np.sqrt(D), seed=77,
        new_token=new_token)


def _run(cfg, **kw):
    hw = H.generate(cfg)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(dw, dev_err=err, **kw)
    code = device_error(err)
    ref, _, _ = oracle.decode_step(hp, hw, threads=8)
    return dw, out, code, ref


@pytest.mark.parametrize("combo", COMBOS, ids=lambda c: "_".join(map(str, c)))
def test_shapes_and_boundaries(combo):
    cfg = _cfg(*combo)
    dw, out, code, ref = _run(cfg)
    assert code == 0
    got = to_f64(out)
    assert_close(got, ref, cfg.name)
    assert np.all(got[0] == 0.0)  # context length 0 -> zeros


def test_new_token_write_then_read():
    cfg = _cfg("bf16", 128, 16, 2, 2, lens=(1, 16, 17, 256, 257, 700), new_token=True)
    _, out, code, ref = _run(cfg)
    assert code == 0
    assert_close(to_f64(out), ref, cfg.name)


def test_oversized_grid_and_workspace_reuse():
    """max_context_len far above the real lengths, and one workspace reused
    by consecutive calls (its counters return to 0)."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = _cfg("f16", 128, 16, 2, 1, lens=(3, 300, 900, 1500))
    hw = H.generate(cfg)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    ref, _, _ = oracle.decode_step(hp, hw)
    mcl = cfg.max_blocks_per_seq * cfg.block_size
    ws = pkv.new_workspace(4, cfg.num_heads, cfg.head_dim, mcl)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        out = run_step(dw, workspace=ws, dev_err=err, max_context_len=mcl)
        assert device_error(err) == 0
        assert_close(to_f64(out), ref, "reuse")
    assert int(ws[: 4 * cfg.num_heads * 4].view(torch.int32).abs().sum()) == 0, "counters not reset"


def test_zero_sequences_is_a_no_op():
    import paged_kv_cache_204_gb300 as pkv
    z = torch.zeros((0, 4, 64), dtype=torch.float16, device="cuda")
    kc = torch.zeros((4, 4, 16, 64), dtype=torch.float16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    cl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    pkv.paged_attention_decode(z, z, kc, kc, bt, cl, 0.1, 16)
    torch.cuda.synchronize()


def test_device_error_bits():
    """Bad indices are reported in the error word and never fault."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = _cfg("f16", 128, 16, 2, 1, lens=(40, 300))
    hw = H.generate(cfg)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # block id out of range
    bt = dw.block_tables.clone()
    bt[1, 2] = cfg.num_blocks + 7
    out = torch.empty_like(dw.q)
    ws = pkv.new_workspace(2, cfg.num_heads, cfg.head_dim, 300)
    pkv.paged_attention_decode(out, dw.q, dw.k_cache, dw.v_cache, bt, dw.context_lens, cfg.scale, 300,
                               workspace=ws, dev_err=err)
    assert device_error(err) & pkv.DEV_ERR_BLOCK_ID
    # context length above max_context_len
    err.zero_()
    ws.zero_()
    pkv.paged_attention_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                               cfg.scale, 100, workspace=pkv.new_workspace(2, cfg.num_heads, 128, 100),
                               dev_err=err)
    assert device_error(err) & pkv.DEV_ERR_CONTEXT_LEN
    # slot out of range, negative slot skipped
    err.zero_()
    k = torch.ones((2, 2, 128), dtype=torch.float16, device="cuda")
    before = dw.k_cache.clone()
    slots = torch.tensor([-1, cfg.num_blocks * cfg.block_size], dtype=torch.int64, device="cuda")
    pkv.reshape_and_cache(k, k, dw.k_cache, dw.v_cache, slots, dev_err=err)
    assert device_error(err) == pkv.DEV_ERR_SLOT
    assert torch.equal(before.view(torch.int16), dw.k_cache.view(torch.int16))
    # pair out of range
    err.zero_()
    pairs = torch.tensor([[0, cfg.num_blocks]], dtype=torch.int64, device="cuda")
    pkv.copy_blocks(dw.k_cache, dw.v_cache, pairs, dev_err=err)
    assert device_error(err) == pkv.DEV_ERR_PAIR
    assert torch.equal(before.view(torch.int16), dw.k_cache.view(torch.int16))


def test_wait_timeout_is_reported_and_context_survives():
    """With a wait limit of 0 every wait that is not already complete gives
    up at once: the kernel reports PKV_DEV_ERR_TIMEOUT, lets its copies land
    and returns; the next call with the default limit is correct."""
    import paged_kv_cache_204_gb300 as pkv
    cfg = synth.get("llama7b")
    hw = H.generate(cfg, num_seqs=16)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = pkv.get_wait_timeout_ns()
    ws = pkv.new_workspace(16, cfg.num_heads, cfg.head_dim, hw.st.max_context_len)
    try:
        pkv.set_wait_timeout_ns(0)
        run_step(dw, workspace=ws, dev_err=err)
        code = device_error(err)
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT
    assert code & ~pkv.DEV_ERR_TIMEOUT == 0
    err.zero_()
    ws.zero_()  # a call that reported a device error may leave counters set
    out = run_step(dw, workspace=ws, dev_err=err)
    assert device_error(err) == 0
    ref, _, _ = oracle.decode_step(hp, hw, threads=8)
    assert_close(to_f64(out), ref, "after timeout")
