"""The allocation-free decode entry point, through the C ABI.

Some callers cannot allocate device memory where they run attention (their
host application owns all device memory, or their memory budget is fixed);
pkv_paged_attention_decode_noalloc serves them with a fixed scratch array
inside the library. Its results must match the workspace entry point's and
the oracle's within the parity tolerance, on consecutive calls that reuse
the same scratch, also after a call that gave up on a wait and left the
scratch's counters set. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as SD
import synth.host as H
from gpu_helpers import ATOL, RTOL, assert_close, to_f64

pytestmark = pytest.mark.gpu


def _host(name, B, **over):
    cfg = synth.get(name).replace(**over)
    return H.generate(cfg, num_seqs=B)


def _workload(name, B, **over):
    return SD.from_host(_host(name, B, **over))


def _close(a, b):
    err = np.abs(a - b)
    assert np.isfinite(a).all() and (err <= ATOL + RTOL * np.abs(b)).all(), float(err.max())


@pytest.mark.parametrize("name,B,over", [
    ("llama13b", 16, {}),                                       # segments split across warps
    ("longctx_bs16", 2, {"num_heads": 4, "num_kv_heads": 4}),  # each segment split many ways
    ("tiny", 4, {}),                                            # fewer tiles than warps
])
def test_noalloc_matches_workspace_entry_point(name, B, over):
    import paged_kv_cache_204_gb300 as pkv
    hw = _host(name, B, **over)
    dw = SD.from_host(hw)
    cfg, st = dw.cfg, dw.st
    mcl = st.max_context_len
    assert pkv.decode_workspace_bytes(st.num_seqs, cfg.num_heads, cfg.head_dim, mcl) <= pkv.NOALLOC_SCRATCH_BYTES
    if dw.slot_mapping.numel():
        pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping)
    ref = torch.empty_like(dw.q)
    ws = pkv.new_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim, mcl)
    pkv.paged_attention_decode(ref, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                               cfg.scale, mcl, workspace=ws)
    ref_np = to_f64(ref)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # two calls in a row share the scratch
        out = torch.full_like(dw.q, float("nan"))
        pkv.paged_attention_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                           dw.context_lens, cfg.scale, mcl, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _close(to_f64(out), ref_np)
    want, _, _ = oracle.decode_step(H.compact_pools(hw), hw, threads=8)
    assert_close(to_f64(out), want, f"noalloc {name}")


def test_noalloc_clears_counters_left_by_a_timed_out_call():
    """A call whose waits run out (wait limit 0) reports PKV_DEV_ERR_TIMEOUT
    and may leave segment counters in the shared scratch set; the next call
    clears the counters it needs before its kernel starts, so it matches the
    workspace entry point and the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    hw = _host("llama13b", 16)
    dw = SD.from_host(hw)
    cfg, st = dw.cfg, dw.st
    mcl = st.max_context_len
    pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = pkv.get_wait_timeout_ns()
    try:
        pkv.set_wait_timeout_ns(0)
        pkv.paged_attention_decode_noalloc(torch.empty_like(dw.q), dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                           dw.context_lens, cfg.scale, mcl, dev_err=err)
        torch.cuda.synchronize()
        code = int(err.item())
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT and code & ~pkv.DEV_ERR_TIMEOUT == 0
    err.zero_()
    out = torch.full_like(dw.q, float("nan"))
    pkv.paged_attention_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                                       cfg.scale, mcl, dev_err=err)
    ref = torch.empty_like(dw.q)
    pkv.paged_attention_decode(ref, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens, cfg.scale,
                               mcl, workspace=pkv.new_workspace(st.num_seqs, cfg.num_heads, cfg.head_dim, mcl))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _close(to_f64(out), to_f64(ref))
    want, _, _ = oracle.decode_step(H.compact_pools(hw), hw, threads=8)
    assert_close(to_f64(out), want, "noalloc after timeout")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import paged_kv_cache_204_gb300 as pkv
    dw = _workload("tiny", 4)
    cfg = dw.cfg
    B, H, D, L = 65535, 128, 128, 8192   # segment counters alone exceed 32 MiB
    assert pkv.decode_workspace_bytes(B, H, D, L) > pkv.NOALLOC_SCRATCH_BYTES
    rc = pkv.lib.pkv_paged_attention_decode_noalloc(
        dw.q.data_ptr(), dw.q.data_ptr(), dw.k_cache.data_ptr(), dw.v_cache.data_ptr(),
        dw.block_tables.data_ptr(), dw.context_lens.data_ptr(), 0.1, H, H, D, cfg.block_size, B,
        L // cfg.block_size, cfg.num_blocks, L, 0, None, None)
    assert rc == pkv.PKV_ERR_WORKSPACE
