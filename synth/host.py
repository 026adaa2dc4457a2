"""Seeded K/V/q values on the host (numpy), for workloads small enough to
generate and check on the CPU.

Values are N(0, 1) * cfg.value_scale, rounded once to the storage type.
Storage convention: fp16/bf16 as raw 16-bit patterns (np.uint16), fp32 as
np.float32. Cache rows that hold no token yet are POISON (all bits set: NaN
in every supported type), so any read of them that reaches a result shows up.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .configs import DecodeConfig
from .structure import Structure, build

POISON16 = np.uint16(0xFFFF)
POISON32_BITS = np.uint32(0xFFFFFFFF)


def storage_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values -> stored elements of `dtype` (round to nearest even)."""
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        # round-to-nearest-even on the 16 dropped bits
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return u.astype(np.uint16)
    raise ValueError(dtype)


def poison(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.full(shape, POISON32_BITS, dtype=np.uint32).view(np.float32)
    return np.full(shape, POISON16, dtype=np.uint16)


def is_poison(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float32:
        return a.view(np.uint32) == POISON32_BITS
    return a == POISON16


@dataclass
class HostWorkload:
    st: Structure
    q: np.ndarray          # [B, H, D]
    prefill_k: np.ndarray  # [U, Hkv, bs, D]: content of st.prefill_blocks (poison past prefill_rows)
    prefill_v: np.ndarray
    new_k: np.ndarray      # [T, Hkv, D]: rows the step writes at st.slot_mapping
    new_v: np.ndarray

    @property
    def cfg(self) -> DecodeConfig:
        return self.st.cfg


def _normal(rng: np.random.Generator, shape, cfg: DecodeConfig) -> np.ndarray:
    return round_to_storage(rng.standard_normal(shape) * cfg.value_scale, cfg.dtype)


def generate(cfg: DecodeConfig, seed: int | None = None, num_seqs: int | None = None,
             st: Structure | None = None) -> HostWorkload:
    seed = cfg.seed if seed is None else seed
    st = build(cfg, seed, num_seqs) if st is None else st
    B, H, Hkv, D, bs = st.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    U, T = st.prefill_blocks.shape[0], st.num_new_tokens
    q = _normal(np.random.default_rng([seed, 10]), (B, H, D), cfg)
    pk = _normal(np.random.default_rng([seed, 11]), (U, Hkv, bs, D), cfg)
    pv = _normal(np.random.default_rng([seed, 12]), (U, Hkv, bs, D), cfg)
    rows = np.arange(bs)[None, :]
    empty = rows >= st.prefill_rows[:, None]            # [U, bs]
    mask = np.broadcast_to(empty[:, None, :, None], pk.shape)
    pk[mask] = poison((), cfg.dtype)
    pv[mask] = poison((), cfg.dtype)
    nk = _normal(np.random.default_rng([seed, 13]), (T, Hkv, D), cfg)
    nv = _normal(np.random.default_rng([seed, 14]), (T, Hkv, D), cfg)
    return HostWorkload(st, q, pk, pv, nk, nv)


@dataclass
class HostPools:
    """Pools holding exactly the blocks a step references, renumbered
    0..n-1 (block ids are opaque: placement does not change results)."""
    k_cache: np.ndarray        # [n, Hkv, bs, D]
    v_cache: np.ndarray
    block_tables: np.ndarray   # int32, renumbered (PAD stays -1)
    slot_mapping: np.ndarray   # int64, renumbered
    copy_pairs: np.ndarray     # int64 [m, 2], renumbered
    ids: np.ndarray            # original id of each compact block
    seqs: np.ndarray           # the sequences these pools serve (rows of block_tables)
    prefix_tables: np.ndarray  # int32, renumbered block tables before the step

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


def compact_pools(w: HostWorkload, seqs: np.ndarray | None = None, fetch=None) -> HostPools:
    """Compact host pools for the whole step, or for a subset of sequences
    (then only their blocks, the copies into them and their new tokens).
    `fetch(ids) -> (k, v)` supplies the pre-step content of physical blocks
    `ids` (default: the workload's prefilled blocks, poison elsewhere)."""
    st, cfg = w.st, w.cfg
    bs = cfg.block_size
    bt = st.block_tables if seqs is None else st.block_tables[seqs]
    pbt = st.prefix_tables if seqs is None else st.prefix_tables[seqs]
    pairs = st.copy_pairs
    if seqs is None:
        ids = st.used_blocks()
    else:
        mine = np.unique(np.concatenate([bt[bt >= 0], pbt[pbt >= 0]])).astype(np.int64)
        if pairs.size:
            pairs = pairs[np.isin(pairs[:, 1], mine)]     # copies into these sequences' blocks
        ids = np.unique(np.concatenate([mine, pairs[:, 0].astype(np.int64)]))
    remap = lambda a: np.searchsorted(ids, a)
    Hkv, D = cfg.num_kv_heads, cfg.head_dim
    if fetch is None:
        kc = poison((ids.shape[0], Hkv, bs, D), cfg.dtype)
        vc = poison((ids.shape[0], Hkv, bs, D), cfg.dtype)
        sel = np.isin(st.prefill_blocks, ids)
        dst = remap(st.prefill_blocks[sel])
        kc[dst] = w.prefill_k[sel]
        vc[dst] = w.prefill_v[sel]
    else:
        kc, vc = fetch(ids)
    bt_c = np.where(bt >= 0, remap(np.maximum(bt, 0)), -1).astype(np.int32)
    pbt_c = np.where(pbt >= 0, remap(np.maximum(pbt, 0)), -1).astype(np.int32)
    sm = st.slot_mapping
    if seqs is not None:
        keep = np.isin(sm // bs, ids)
        sm = np.where(keep, sm, -1)   # tokens of other sequences become padding
    sm_c = np.where(sm >= 0, remap(np.maximum(sm, 0) // bs) * bs + np.maximum(sm, 0) % bs, -1)
    pairs_c = remap(pairs).astype(np.int64).reshape(-1, 2)
    rows = np.arange(st.num_seqs) if seqs is None else np.asarray(seqs)
    return HostPools(kc, vc, bt_c, sm_c.astype(np.int64), pairs_c, ids, rows, pbt_c)


def full_pools(w: HostWorkload) -> tuple[np.ndarray, np.ndarray]:
    """Pools of cfg.num_blocks blocks (poison except prefilled rows). Only for
    small pools."""
    cfg = w.cfg
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    kc, vc = poison(shape, cfg.dtype), poison(shape, cfg.dtype)
    kc[w.st.prefill_blocks] = w.prefill_k
    vc[w.st.prefill_blocks] = w.prefill_v
    return kc, vc
