"""Named synthetic decode workloads.

Each preset fixes shapes, the length distribution, the physical pool size, the
element type, the value distribution and a seed. They stand in for the
ShareGPT-derived request mix of the pages' evaluation ("PagedAttention: the KV
cache was the bottleneck all along", section "The number that made us read the
code": LLaMA-7B and LLaMA-13B serving), using LLaMA-shaped heads and
lognormal/uniform context lengths.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int           # running sequences (for "cow": prompts * samples)
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str              # "f32" | "f16" | "bf16"
    num_blocks: int         # physical blocks in each pool
    lengths: tuple          # ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("fixed", (..))
    value_scale: float      # K, V, q values are N(0, 1) * value_scale, rounded to dtype
    scale: float            # softmax scale applied to q . k
    seed: int
    new_token: bool = False         # the step also writes each sequence's newest K/V row
    samples: int = 1                # "cow": completions per prompt sharing the prompt's blocks
    tail: tuple | None = None       # "cow": ("uniform", lo, hi) divergent tail tokens per sample

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_len(self) -> int:
        """Largest context length the distribution can produce."""
        top = lambda spec: max(spec[1]) if spec[0] == "fixed" else spec[-1]
        hi = top(self.lengths)
        if self.tail is not None:
            hi += top(self.tail)
        return int(hi)

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_len // self.block_size)

    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token across all kv heads (one layer)."""
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    def replace(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


INV_SQRT_128 = 1.0 / math.sqrt(128.0)

PRESETS: dict[str, DecodeConfig] = {
    # Tiny paged decode: fp32, 64 blocks handed out in a random permutation.
    "tiny": DecodeConfig("tiny", num_seqs=4, num_heads=2, num_kv_heads=2, head_dim=64,
                         block_size=16, dtype="f32", num_blocks=64,
                         lengths=("uniform", 1, 100), value_scale=1.0, scale=1.0 / 8.0,
                         seed=2041),
    # LLaMA-7B-shaped step: values N(0,1)/sqrt(128) in fp16, scale 1/sqrt(128).
    "llama7b": DecodeConfig("llama7b", num_seqs=64, num_heads=32, num_kv_heads=32,
                            head_dim=128, block_size=16, dtype="f16", num_blocks=40000,
                            lengths=("lognormal", 300, 1.0, 16, 2048), value_scale=INV_SQRT_128,
                            scale=INV_SQRT_128, seed=2042),
    # LLaMA-13B-shaped step (the headline workload): bf16, plus the write of
    # each sequence's newest K/V row before attention reads it.
    "llama13b": DecodeConfig("llama13b", num_seqs=128, num_heads=40, num_kv_heads=40,
                             head_dim=128, block_size=16, dtype="bf16", num_blocks=40000,
                             lengths=("lognormal", 500, 1.0, 16, 2048), value_scale=1.0,
                             scale=INV_SQRT_128, seed=2043, new_token=True),
    # Parallel sampling: 32 prompts x 3 samples share ref-counted prompt blocks,
    # diverge by 1..256 tail tokens; the shared partial block is copied on write.
    "cow": DecodeConfig("cow", num_seqs=96, num_heads=40, num_kv_heads=40, head_dim=128,
                        block_size=16, dtype="f16", num_blocks=40000,
                        lengths=("uniform", 128, 1024), value_scale=1.0, scale=INV_SQRT_128,
                        seed=2044, samples=3, tail=("uniform", 1, 256)),
}
# Long-context split decode, one preset per block size of the sweep.
for _bs in (8, 16, 32):
    PRESETS[f"longctx_bs{_bs}"] = DecodeConfig(
        f"longctx_bs{_bs}", num_seqs=8, num_heads=32, num_kv_heads=32, head_dim=128,
        block_size=_bs, dtype="f16", num_blocks=200000, lengths=("uniform", 16384, 32768),
        value_scale=1.0, scale=INV_SQRT_128, seed=2045 + _bs)


def get(name: str) -> DecodeConfig:
    return PRESETS[name]
