"""Helpers for the GPU parity tests: run a decode step through the C ABI and
compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth.host as H
from synth.device import DeviceWorkload, to_storage

# Tolerance for fp16/bf16 (and fp32) attention outputs with fp32 accumulation:
# an element passes if |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL, RTOL = 2e-3, 1e-2


def run_step(dw: DeviceWorkload, workspace=None, dev_err=None, max_context_len=None,
             out=None) -> torch.Tensor:
    """The step's order: copy-on-write copies, new K/V rows, attention."""
    import paged_kv_cache_204_gb300 as pkv
    st = dw.st
    if dw.copy_pairs.numel():
        pkv.copy_blocks(dw.k_cache, dw.v_cache, dw.copy_pairs, dev_err=dev_err)
    if dw.slot_mapping.numel():
        pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=dev_err)
    mcl = st.max_context_len if max_context_len is None else max_context_len
    if out is None:
        out = torch.empty_like(dw.q)
    if workspace is None:
        workspace = pkv.new_workspace(st.num_seqs, dw.cfg.num_heads, dw.cfg.head_dim, mcl, dw.q.device)
    pkv.paged_attention_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                               dw.cfg.scale, mcl, workspace=workspace, dev_err=dev_err)
    return out


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    big = np.abs(ref) > 1e-2
    stats = {"max_abs": float(err.max(initial=0.0)),
             "max_rel": float((err[big] / np.abs(ref[big])).max(initial=0.0)),
             "n": int(ref.size), "n_bad": int(bad.sum())}
    assert not bad.any(), f"{what}: {stats}"
    return stats


def host_view(dw: DeviceWorkload) -> H.HostWorkload:
    """q and the step's new rows on the host (pools stay on the device)."""
    return H.HostWorkload(dw.st, to_storage(dw.q), None, None, to_storage(dw.new_k), to_storage(dw.new_v))


def sample_pools(dw: DeviceWorkload, seqs) -> H.HostPools:
    """Host copies of the pre-step content of every block the given sequences
    use. Call BEFORE any kernel touches the pools."""
    dev = dw.k_cache.device

    def fetch(ids):
        idx = torch.from_numpy(ids).to(dev)
        return to_storage(dw.k_cache[idx]), to_storage(dw.v_cache[idx])

    return H.compact_pools(host_view(dw), np.asarray(seqs), fetch=fetch)


def oracle_outputs(dw: DeviceWorkload, hp: H.HostPools, threads: int = 8) -> np.ndarray:
    """Oracle step for the sequences hp serves; rows in hp.seqs order."""
    out, _, _ = oracle.decode_step(hp, host_view(dw), threads=threads)
    return out


def device_error(err: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(err.item())
