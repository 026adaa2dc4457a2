"""Seeded K/V/q values generated directly in device memory (torch), for
full-size workloads whose pools (tens of GB) are too large to build on the
host. Same structure as host.py (synth.structure.build), same value
distribution (N(0, 1) * value_scale rounded to the storage type), drawn by a
seeded torch generator on the device; every cache row that holds no token is
POISON (all bits set).

Only torch tensor plumbing lives here (random fill, index copies of whole
prefilled blocks, poison fill); none of the decode arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from .configs import DecodeConfig
from .structure import Structure, build

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
BITS_DTYPE = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}


@dataclass
class DeviceWorkload:
    st: Structure
    q: torch.Tensor             # [B, H, D]
    k_cache: torch.Tensor       # [num_blocks, Hkv, bs, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor  # int32 [B, MB]
    context_lens: torch.Tensor  # int32 [B]
    new_k: torch.Tensor         # [T, Hkv, D]
    new_v: torch.Tensor
    slot_mapping: torch.Tensor  # int64 [T]
    copy_pairs: torch.Tensor    # int64 [n, 2]

    @property
    def cfg(self) -> DecodeConfig:
        return self.st.cfg


def _randn(shape, cfg: DecodeConfig, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if cfg.value_scale != 1.0:
        x.mul_(cfg.value_scale)
    return x.to(TORCH_DTYPE[cfg.dtype])


def fill_poison(t: torch.Tensor) -> None:
    t.view(torch.uint8).fill_(0xFF)


def generate(cfg: DecodeConfig, device="cuda", seed: int | None = None,
             num_seqs: int | None = None, st: Structure | None = None,
             chunk_blocks: int = 4096) -> DeviceWorkload:
    seed = cfg.seed if seed is None else seed
    st = build(cfg, seed, num_seqs) if st is None else st
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed) * 1000003 + 17)
    B, H, Hkv, D, bs = st.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    shape = (cfg.num_blocks, Hkv, bs, D)
    kc = torch.empty(shape, dtype=TORCH_DTYPE[cfg.dtype], device=dev)
    vc = torch.empty(shape, dtype=TORCH_DTYPE[cfg.dtype], device=dev)
    fill_poison(kc)
    fill_poison(vc)
    pb = torch.from_numpy(st.prefill_blocks).to(dev)
    pr = torch.from_numpy(st.prefill_rows.astype(np.int64)).to(dev)
    rows = torch.arange(bs, device=dev)
    for cache in (kc, vc):
        for a in range(0, pb.shape[0], chunk_blocks):
            ids = pb[a:a + chunk_blocks]
            vals = _randn((ids.shape[0], Hkv, bs, D), cfg, gen, dev)
            empty = (rows[None, :] >= pr[a:a + chunk_blocks, None])[:, None, :, None]
            bits = vals.view(BITS_DTYPE[cfg.dtype])
            bits.masked_fill_(empty.expand_as(bits), -1)   # poison rows past the prefill
            cache[ids] = vals
    q = _randn((B, H, D), cfg, gen, dev)
    T = st.num_new_tokens
    nk = _randn((T, Hkv, D), cfg, gen, dev)
    nv = _randn((T, Hkv, D), cfg, gen, dev)
    return DeviceWorkload(
        st=st, q=q, k_cache=kc, v_cache=vc,
        block_tables=torch.from_numpy(st.block_tables).to(dev),
        context_lens=torch.from_numpy(st.context_lens).to(dev),
        new_k=nk, new_v=nv,
        slot_mapping=torch.from_numpy(st.slot_mapping).to(dev),
        copy_pairs=torch.from_numpy(st.copy_pairs).to(dev).reshape(-1, 2).contiguous())


def from_host(hw, device="cuda") -> DeviceWorkload:
    """Upload a synth.host.HostWorkload into full-size device pools (the
    prefilled blocks at their physical ids, poison elsewhere)."""
    st, cfg = hw.st, hw.cfg
    dev = torch.device(device)
    td = TORCH_DTYPE[cfg.dtype]

    def up(a: np.ndarray) -> torch.Tensor:
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a if cfg.dtype == "f32" else a.view(np.int16))
        return t.to(dev).view(td)

    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    kc = torch.empty(shape, dtype=td, device=dev)
    vc = torch.empty(shape, dtype=td, device=dev)
    fill_poison(kc)
    fill_poison(vc)
    pb = torch.from_numpy(st.prefill_blocks).to(dev)
    if pb.numel():
        kc[pb] = up(hw.prefill_k)
        vc[pb] = up(hw.prefill_v)
    return DeviceWorkload(
        st=st, q=up(hw.q), k_cache=kc, v_cache=vc,
        block_tables=torch.from_numpy(st.block_tables).to(dev),
        context_lens=torch.from_numpy(st.context_lens).to(dev),
        new_k=up(hw.new_k), new_v=up(hw.new_v),
        slot_mapping=torch.from_numpy(st.slot_mapping).to(dev),
        copy_pairs=torch.from_numpy(st.copy_pairs).to(dev).reshape(-1, 2).contiguous())


def to_storage(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host numpy in the oracle's storage convention."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)
