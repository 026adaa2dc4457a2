"""The allocation-free decode entry point, through the C ABI.

Some callers cannot allocate device memory where they run attention (their
host application owns all device memory, or their memory budget is fixed);
pkv_paged_attention_decode_noalloc serves them with a fixed scratch array
inside the library. Its results must match the workspace entry point's
within the parity tolerance, on consecutive calls that reuse the same
scratch. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
import synth.device as SD
import synth.host as H
from gpu_helpers import ATOL, RTOL, to_f64

pytestmark = pytest.mark.gpu


def _workload(name, B, **over):
    cfg = synth.get(name).replace(**over)
    return SD.from_host(H.generate(cfg, num_seqs=B))


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
    dw = _workload(name, B, **over)
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
