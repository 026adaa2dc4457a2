"""Seeded synthetic beam-search decoding workloads.

Beam search keeps `width` beams per request; at every step each new beam
continues one of the current beams, so beams share long prefixes and are
forked and discarded all the time ("PagedAttention: the KV cache was the
bottleneck all along", section "Virtual memory for attention"). There is no
model here: which beam each new beam continues is drawn from a seeded,
skewed distribution (better-ranked beams are continued more often), and the
K/V rows and queries are N(0, 1) * value_scale rounded to the storage type.

Holds shapes, lengths, parent choices and random values only: none of the
attention or cache arithmetic.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np

from .host import round_to_storage
from .structure import draw_lengths


@dataclass(frozen=True)
class BeamConfig:
    name: str
    requests: int
    width: int              # beams per request
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    num_blocks: int
    prompt: tuple           # prompt length distribution (see structure.draw_lengths)
    steps: int              # decode steps the workload runs (and the pool is sized for)
    value_scale: float
    scale: float
    seed: int

    @property
    def num_seqs(self) -> int:
        return self.requests * self.width

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_len(self) -> int:
        return int(self.prompt[-1]) + self.steps

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_len // self.block_size)

    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    def replace(self, **kw) -> "BeamConfig":
        return dataclasses.replace(self, **kw)


PRESETS = {
    # parity-test size: grouped-query heads, block boundaries every 8 tokens
    "beam_small": BeamConfig("beam_small", requests=3, width=4, num_heads=4, num_kv_heads=2, head_dim=64,
                             block_size=8, dtype="f16", num_blocks=400, prompt=("uniform", 5, 60), steps=12,
                             value_scale=1.0, scale=1.0 / 8.0, seed=2051),
    # benchmark size: LLaMA-13B-shaped heads, beam width 4, prompts as in the copy-on-write workload
    "beam": BeamConfig("beam", requests=16, width=4, num_heads=40, num_kv_heads=40, head_dim=128,
                       block_size=16, dtype="f16", num_blocks=40000, prompt=("uniform", 128, 1024), steps=256,
                       value_scale=1.0, scale=1.0 / math.sqrt(128), seed=2052),
}


def get(name: str) -> BeamConfig:
    return PRESETS[name]


def prompt_lengths(cfg: BeamConfig) -> np.ndarray:
    return draw_lengths(cfg.prompt, cfg.requests, np.random.default_rng([cfg.seed, 1]))


def parent_stream(cfg: BeamConfig):
    """Yields, step after step, the parent choice of every request:
    int32 [requests][width], row r's entry i = the beam new beam i continues.
    Beam rank j is continued with probability proportional to (width - j)^2."""
    rng = np.random.default_rng([cfg.seed, 3])
    W = cfg.width
    p = np.arange(W, 0, -1, dtype=np.float64) ** 2
    p /= p.sum()
    while True:
        yield rng.choice(W, size=(cfg.requests, W), p=p).astype(np.int32)


class HostValues:
    """Seeded host values (storage patterns) for small beam workloads:
    prompt rows of each request and, per step, the new K/V row of every new
    beam and every new beam's query."""

    def __init__(self, cfg: BeamConfig):
        self.cfg = cfg
        self._rng = np.random.default_rng([cfg.seed, 4])

    def _normal(self, shape) -> np.ndarray:
        return round_to_storage(self._rng.standard_normal(shape) * self.cfg.value_scale, self.cfg.dtype)

    def prompt(self, length: int) -> tuple[np.ndarray, np.ndarray]:
        c = self.cfg
        return self._normal((length, c.num_kv_heads, c.head_dim)), self._normal((length, c.num_kv_heads, c.head_dim))

    def step(self) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """(new_k, new_v [B, Hkv, D], q [B, H, D]) for one step, B = requests * width."""
        c = self.cfg
        B = c.num_seqs
        k = self._normal((B, c.num_kv_heads, c.head_dim))
        v = self._normal((B, c.num_kv_heads, c.head_dim))
        q = self._normal((B, c.num_heads, c.head_dim))
        return k, v, q
