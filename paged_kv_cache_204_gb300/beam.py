"""Beam-search decoding over the paged KV cache.

Beams of one request share their common prefix in the cache and are forked
and discarded at every step ("PagedAttention: the KV cache was the
bottleneck all along", section "Virtual memory for attention"). One step:

  host   the library's block manager ends the beams nobody continues, forks
         the ones continued more than once, and reserves a slot for every new
         beam's token (copy-on-write pairs for shared partly filled blocks);
         block tables, context lengths and each request's shared prefix are
         exported in the decode kernels' layout;
  device copy_blocks (the copy-on-write pairs), reshape_and_cache (the new
         beams' K/V rows), then the grouped decode kernel with one group per
         request, so the request's shared prefix is read once for all beams.

This module only marshals: the bookkeeping runs in the C++ block manager and
every byte of K/V is moved and read by the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (copy_blocks, new_grouped_workspace, paged_attention_decode_grouped, reshape_and_cache)
from .block_manager import BlockManager


@dataclass
class StepPlan:
    """Host arrays of one step, batch order = request-major, beam-minor."""
    seqs: np.ndarray           # int32 [B]   sequence ids of the new beams
    slots: np.ndarray          # int64 [B]   cache slot of each new beam's token
    copy_pairs: np.ndarray     # int64 [k,2] blocks to copy before the writes
    block_tables: np.ndarray   # int32 [B, max_blocks_per_seq]
    context_lens: np.ndarray   # int32 [B]
    group_start: np.ndarray    # int32 [R+1]
    shared_blocks: np.ndarray  # int32 [R]
    max_context_len: int


@dataclass
class DevicePlan:
    slots: torch.Tensor
    copy_pairs: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    group_start: torch.Tensor
    shared_blocks: torch.Tensor
    max_context_len: int


_FIELDS = ("slots", "copy_pairs", "block_tables", "context_lens", "group_start", "shared_blocks")


class BeamDecoder:
    """Beam search of `width` beams per request over caches k_cache, v_cache
    ([num_blocks, Hkv, block_size, D], on the GPU)."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, width: int, max_blocks_per_seq: int,
                 seed: int = 0):
        self.k_cache, self.v_cache = k_cache, v_cache
        nb, _, bs, _ = k_cache.shape
        self.width = int(width)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        self.block_size = bs
        self.manager = BlockManager(nb, bs, seed=seed)
        self.requests: list[list[int]] = []
        self._ws = None
        self._ws_key = None
        self._pinned: dict[str, torch.Tensor] = {}
        self._dev: dict[str, torch.Tensor] = {}
        self._staged = None  # event: the last upload's copies have read the pinned buffers

    # -- requests ---------------------------------------------------------------
    def admit(self, prompt_len: int) -> np.ndarray:
        """Host part of add_request: a new request of `width` beams sharing a
        prompt of prompt_len tokens; returns the prompt rows' slots (int64)."""
        s = self.manager.add_seq()
        slots, _ = self.manager.append(s, int(prompt_len))
        self.requests.append([s] + [self.manager.fork(s) for _ in range(self.width - 1)])
        return slots

    def add_request(self, prompt_k: torch.Tensor, prompt_v: torch.Tensor, dev_err=None, stream=None) -> int:
        """Write a prompt's K/V rows ([P, Hkv, D], on the GPU) into fresh
        blocks and start the request with `width` beams that share them."""
        slots = self.admit(prompt_k.shape[0])
        if prompt_k.shape[0]:
            dev_slots = torch.from_numpy(slots).to(prompt_k.device, non_blocking=False)
            reshape_and_cache(prompt_k, prompt_v, self.k_cache, self.v_cache, dev_slots, dev_err=dev_err,
                              stream=stream)
        return len(self.requests) - 1

    # -- one step ---------------------------------------------------------------------
    def plan(self, parents) -> StepPlan:
        """Host bookkeeping of one step: parents [R][W], entry (r, i) = the
        current beam of request r that new beam i continues."""
        R = len(self.requests)
        parents = np.asarray(parents, dtype=np.int32).reshape(R, self.width)
        beams = np.asarray(self.requests, dtype=np.int32).reshape(R, self.width)
        new, slots, pairs, shared = self.manager.beam_step_many(beams, parents, 1)
        self.requests = new.tolist()
        seqs = new.reshape(-1)
        bt, cl = self.manager.export(seqs, self.max_blocks_per_seq)
        return StepPlan(seqs=seqs, slots=slots, copy_pairs=pairs,
                        block_tables=bt, context_lens=cl,
                        group_start=(np.arange(R + 1, dtype=np.int32) * self.width),
                        shared_blocks=shared,
                        max_context_len=int(cl.max()) if cl.size else 0)

    def _buffer(self, table: dict, name: str, nbytes: int, pinned: bool) -> torch.Tensor:
        buf = table.get(name)
        if buf is None or buf.numel() < nbytes:
            n = max(256, 1 << (max(nbytes, 1) - 1).bit_length())
            buf = (torch.empty(n, dtype=torch.uint8).pin_memory() if pinned
                   else torch.empty(n, dtype=torch.uint8, device=self.k_cache.device))
            table[name] = buf
        return buf

    def upload(self, plan: StepPlan, stream=None) -> DevicePlan:
        """Copy a plan to the device in one transfer: every array is packed
        (16-byte aligned) into one reused pinned staging buffer, copied into
        one reused device buffer, and returned as views of it. The views stay
        valid until the next upload, which the stream orders after the work
        already queued on them."""
        stream = torch.cuda.current_stream(self.k_cache.device) if stream is None else stream
        if self._staged is not None:
            self._staged.synchronize()  # the previous transfer has left the staging buffer
        arrays, offsets, total = [], [], 0
        for name in _FIELDS:
            a = np.ascontiguousarray(getattr(plan, name))
            arrays.append(a)
            offsets.append(total)
            total += (a.nbytes + 15) & ~15
        host = self._buffer(self._pinned, "plan", total, pinned=True)
        dev = self._buffer(self._dev, "plan", total, pinned=False)
        hv = host.numpy()
        for a, o in zip(arrays, offsets):
            hv[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
        out = {}
        with torch.cuda.stream(stream):
            if total:
                dev[:total].copy_(host[:total], non_blocking=True)
            self._staged = torch.cuda.Event()
            self._staged.record(stream)
        for name, a, o in zip(_FIELDS, arrays, offsets):
            t = dev[o:o + a.nbytes].view(torch.from_numpy(a[:0].reshape(-1)).dtype)
            out[name] = t.view(a.shape)
        return DevicePlan(max_context_len=plan.max_context_len, **out)

    def workspace(self, num_heads: int, head_dim: int) -> torch.Tensor:
        B, R = len(self.requests) * self.width, len(self.requests)
        key = (B, num_heads, head_dim, R)
        if self._ws_key != key:
            self._ws = new_grouped_workspace(B, num_heads, head_dim, 0, R, device=self.k_cache.device)
            self._ws_key = key
        return self._ws

    def run(self, dp: DevicePlan, new_k: torch.Tensor, new_v: torch.Tensor, q: torch.Tensor, scale: float,
            out: torch.Tensor, dev_err=None, stream=None) -> torch.Tensor:
        """Device part of a step: copies, the new rows, grouped attention.
        new_k, new_v [B, Hkv, D] and q, out [B, H, D] in the plan's order."""
        ws = self.workspace(q.shape[1], q.shape[2])
        if dp.copy_pairs.numel():
            copy_blocks(self.k_cache, self.v_cache, dp.copy_pairs, dev_err=dev_err, stream=stream)
        reshape_and_cache(new_k, new_v, self.k_cache, self.v_cache, dp.slots, dev_err=dev_err, stream=stream)
        paged_attention_decode_grouped(out, q, self.k_cache, self.v_cache, dp.block_tables, dp.context_lens, scale,
                                       dp.max_context_len, dp.group_start, dp.shared_blocks, ws, dev_err=dev_err,
                                       stream=stream)
        return out

    def step(self, parents, new_k: torch.Tensor, new_v: torch.Tensor, q: torch.Tensor, scale: float,
             out: torch.Tensor | None = None, dev_err=None, stream=None) -> torch.Tensor:
        """plan + upload + run."""
        out = torch.empty_like(q) if out is None else out
        return self.run(self.upload(self.plan(parents), stream=stream), new_k, new_v, q, scale, out,
                        dev_err=dev_err, stream=stream)
