"""Seeded synthetic prefill workloads with a system prompt shared by users.

"PagedAttention: the KV cache was the bottleneck all along", section "What is
left": shared blocks for common system prompts across users. A root sequence
holds the system prompt; every user forks it (sharing its blocks) and
appends its own prompt; the user's tokens are the queries of one prefill
step, attending causally to the system prompt and to their own earlier
tokens. The system prompt's last block, when partly filled, is copied on
write by the users that append into it.

Holds shapes, lengths, block placement and random values only: none of the
attention or cache arithmetic.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np

from .blockmgr import BlockManager
from .host import poison, round_to_storage
from .structure import PAD_BLOCK, draw_lengths


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    users: int
    system_len: int         # tokens of the shared system prompt (0: no sharing)
    user_len: tuple         # length distribution of each user's prompt (structure.draw_lengths)
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    num_blocks: int
    value_scale: float
    scale: float
    seed: int

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_len(self) -> int:
        top = max(self.user_len[1]) if self.user_len[0] == "fixed" else self.user_len[-1]
        return self.system_len + int(top)

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_len // self.block_size)

    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    def replace(self, **kw) -> "PrefillConfig":
        return dataclasses.replace(self, **kw)


PRESETS = {
    "prefill_small": PrefillConfig("prefill_small", users=3, system_len=37, user_len=("uniform", 1, 90),
                                   num_heads=4, num_kv_heads=2, head_dim=64, block_size=8, dtype="f16",
                                   num_blocks=200, value_scale=1.0, scale=1.0 / 8.0, seed=2081),
    # LLaMA-13B-shaped heads; a 1024-token system prompt shared by 16 users with 256..768-token prompts
    "prefill": PrefillConfig("prefill", users=16, system_len=1024, user_len=("uniform", 256, 768),
                             num_heads=40, num_kv_heads=40, head_dim=128, block_size=16, dtype="bf16",
                             num_blocks=40000, value_scale=1.0, scale=1.0 / math.sqrt(128), seed=2082),
    # the same step over binary16 caches and queries
    "prefill_f16": PrefillConfig("prefill_f16", users=16, system_len=1024, user_len=("uniform", 256, 768),
                                 num_heads=40, num_kv_heads=40, head_dim=128, block_size=16, dtype="f16",
                                 num_blocks=40000, value_scale=1.0, scale=1.0 / math.sqrt(128), seed=2082),
}


def get(name: str) -> PrefillConfig:
    return PRESETS[name]


@dataclass
class PrefillLayout:
    cfg: PrefillConfig
    system_slots: np.ndarray   # int64 [system_len]: where the system prompt's rows go
    copy_pairs: np.ndarray     # int64 [k, 2]: copy-on-write of the system prompt's partly filled block
    user_slots: np.ndarray     # int64 [total_queries]: the users' rows, user after user
    block_tables: np.ndarray   # int32 [users, max_blocks_per_seq], PAD_BLOCK past the end
    context_lens: np.ndarray   # int32 [users]: system_len + own prompt
    query_start: np.ndarray    # int32 [users + 1]
    max_query_len: int

    @property
    def total_queries(self) -> int:
        return int(self.query_start[-1])


def build(cfg: PrefillConfig, seed: int | None = None) -> PrefillLayout:
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng([seed, 1])
    lens = draw_lengths(cfg.user_len, cfg.users, rng)
    mgr = BlockManager(cfg.num_blocks, cfg.block_size, np.random.default_rng([seed, 2]))
    root = mgr.new_seq()
    sys_slots = np.array(mgr.append(root, cfg.system_len), dtype=np.int64)
    users = [mgr.fork(root) for _ in range(cfg.users)]
    mgr.free_seq(root)
    user_slots = []
    for u, s in enumerate(users):
        user_slots += mgr.append(s, int(lens[u]))
    MB = cfg.max_blocks_per_seq
    bt = np.full((cfg.users, MB), PAD_BLOCK, dtype=np.int32)
    cl = np.zeros(cfg.users, dtype=np.int32)
    for u, s in enumerate(users):
        t = mgr.tables[s]
        bt[u, :len(t)] = t
        cl[u] = mgr.lengths[s]
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return PrefillLayout(cfg=cfg, system_slots=sys_slots,
                         copy_pairs=np.array(mgr.cow_pairs, dtype=np.int64).reshape(-1, 2),
                         user_slots=np.array(user_slots, dtype=np.int64), block_tables=bt, context_lens=cl,
                         query_start=qs, max_query_len=int(lens.max()) if lens.size else 0)


@dataclass
class PrefillValues:
    """Host values (storage patterns): system prompt rows, the users' rows
    (user after user) and the users' queries."""
    system_k: np.ndarray   # [system_len, Hkv, D]
    system_v: np.ndarray
    user_k: np.ndarray     # [total_queries, Hkv, D]
    user_v: np.ndarray
    q: np.ndarray          # [total_queries, H, D]


def host_values(cfg: PrefillConfig, layout: PrefillLayout, seed: int | None = None) -> PrefillValues:
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng([seed, 3])
    n = layout.total_queries
    nrm = lambda shape: round_to_storage(rng.standard_normal(shape) * cfg.value_scale, cfg.dtype)
    return PrefillValues(system_k=nrm((cfg.system_len, cfg.num_kv_heads, cfg.head_dim)),
                         system_v=nrm((cfg.system_len, cfg.num_kv_heads, cfg.head_dim)),
                         user_k=nrm((n, cfg.num_kv_heads, cfg.head_dim)), user_v=nrm((n, cfg.num_kv_heads, cfg.head_dim)),
                         q=nrm((n, cfg.num_heads, cfg.head_dim)))


def host_pools(cfg: PrefillConfig) -> tuple[np.ndarray, np.ndarray]:
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    return poison(shape, cfg.dtype), poison(shape, cfg.dtype)
