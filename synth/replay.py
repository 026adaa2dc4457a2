"""Drive a block manager through the allocation steps of a workload.

Any object with add_seq() (or new_seq()), fork(seq) and append(seq, n) works:
the library's host block manager, the oracle's block model, or this
package's own layout manager. The lengths are the draws
synth.structure.build makes for the same workload and seed, so the replayed
state is that workload's KV cache at its decode step. This module holds no
allocation logic of its own.
"""
from __future__ import annotations

import numpy as np

from .configs import DecodeConfig
from .structure import draw_lengths


def replay(mgr, cfg: DecodeConfig, seed: int | None = None, num_seqs: int | None = None) -> list[int]:
    """Sequence handles of the workload's batch, in batch order, after:
    copy-on-write workloads — each prompt appended to a new sequence, forked
    into its samples, then every sample's tail appended in batch order;
    others — each sequence appended to its full context length."""
    seed = cfg.seed if seed is None else seed
    B = cfg.num_seqs if num_seqs is None else num_seqs
    rng = np.random.default_rng([seed, 1])
    add = getattr(mgr, "add_seq", None) or mgr.new_seq
    if cfg.samples > 1:
        if B % cfg.samples:
            raise ValueError("num_seqs must be a multiple of samples")
        prompts = B // cfg.samples
        plen = draw_lengths(cfg.lengths, prompts, rng)
        tails = draw_lengths(cfg.tail, B, rng)
        order = []
        for p in range(prompts):
            root = add()
            mgr.append(root, int(plen[p]))
            order += [root] + [mgr.fork(root) for _ in range(cfg.samples - 1)]
        for i, s in enumerate(order):
            mgr.append(s, int(tails[i]))
        return order
    lens = draw_lengths(cfg.lengths, B, rng)
    order = []
    for i in range(B):
        s = add()
        mgr.append(s, int(lens[i]))
        order.append(s)
    return order
