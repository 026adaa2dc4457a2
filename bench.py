#!/usr/bin/env python
"""Benchmark of the paged decode hot path on the LLaMA-13B-shaped workload.

One step = one layer's decode step of the workload: reshape_and_cache of the
128 new K/V rows into their cache slots, then paged decode attention of the
128 query tokens (40 heads, head_dim 128, bf16) over their 16..2048-token
contexts scattered through a 40 000-block pool. Inputs are seeded synthetic
data resident in HBM; L2 is flushed (256 MiB written, another 256 MiB read) between timed steps and
each step is timed with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--attention plain|grouped]

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica
of the workload (different seed): weak scaling, no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attention KV GB/s and % of HBM roofline; sequences/s per decode step"
WORKLOAD = "llama13b"
CSRC = os.path.join(ROOT, "paged_kv_cache_204_gb300", "csrc")
# committed ncu summaries that record a kernel's DRAM bytes per launch, keyed by
# a hash of the kernel sources they were taken on
PROFILES = {
    "plain": (os.path.join(ROOT, "profiles", "pa_decode_llama13b.md"), ("decode.cuh",)),
    "fp8": (os.path.join(ROOT, "profiles", "pa_decode_fp8_llama13b.md"), ("decode.cuh",)),
    "q4": (os.path.join(ROOT, "profiles", "pa_decode_q4_0_llama13b.md"), ("decode.cuh",)),
    "grouped": (os.path.join(ROOT, "profiles", "pa_decode_grouped_cow.md"), ("decode.cuh", "decode_grouped.cuh")),
}
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def workload_bytes(st, kv_elem_bytes: int | None = None, new_rows: int | None = None,
                   copy_pairs: int | None = None, kv_row_bytes: int | None = None) -> dict:
    """Algorithmic bytes of one step: attention reads each distinct cached
    (block, row) once for K and once for V plus q, and writes out; the cache
    write reads the new rows and writes them into the pools; each
    copy-on-write pair reads and writes one whole block of both pools.
    new_rows / copy_pairs: the step's counts when they differ from the
    structure's (a copy-on-write decode step writes one row per sample).
    kv_row_bytes: bytes of one cached row of head_dim values when they are
    not head_dim elements (q4_0 rows)."""
    cfg = st.cfg
    es = cfg.elem_bytes
    kes = es if kv_elem_bytes is None else kv_elem_bytes  # cached element (1 for fp8 pools)
    head_row = cfg.head_dim * kes if kv_row_bytes is None else kv_row_bytes
    row = cfg.num_kv_heads * head_row                    # one token, one of K/V, all kv heads, as cached
    qo = st.num_seqs * cfg.num_heads * cfg.head_dim * es
    attn = 2 * st.unique_kv_tokens() * row + 2 * qo
    n_new = st.num_new_tokens if new_rows is None else new_rows
    n_pairs = st.copy_pairs.shape[0] if copy_pairs is None else copy_pairs
    cache_write = 2 * n_new * (cfg.num_kv_heads * cfg.head_dim * es + row)  # read the new rows, write them cached
    copies = 2 * 2 * n_pairs * cfg.block_size * row
    return {"attention": attn, "cache_write": cache_write, "copy": copies,
            "step": attn + cache_write + copies}


def step_counts(cfg, st) -> dict:
    """New rows and copy pairs of one timed step: a copy-on-write decode step
    writes each sample's newest row (its tail and the copies at divergence
    are history); other workloads write the structure's new rows."""
    if cfg.samples > 1:
        return {"new_rows": st.num_seqs, "copy_pairs": 0}
    return {}


def describe_lengths(spec) -> str:
    if spec[0] == "lognormal":
        return f"lognormal(median {spec[1]}, sigma {spec[2]}) clipped to [{spec[3]}, {spec[4]}]"
    if spec[0] == "uniform":
        return f"uniform in [{spec[1]}, {spec[2]}]"
    return f"fixed {list(spec[1])}"


def flush_desc(mode: str = "write+read") -> str:
    if mode == "write+read":
        return (f"flushed between timed steps: {FLUSH_BYTES >> 20} MiB written, then another "
                f"{FLUSH_BYTES >> 20} MiB read (the flush's dirty lines reach HBM before the step)")
    return f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB write)"


def config_json(cfg, st, world: int, attention: str = "plain", kv: str | None = None,
                flush: str = "write+read") -> dict:
    parts = [f"{cfg.name}-shaped decode step: {st.num_seqs} seqs, {cfg.num_heads} heads "
             f"({cfg.num_kv_heads} kv), head_dim {cfg.head_dim}, block_size {cfg.block_size}, "
             f"{cfg.dtype} storage with fp32 accumulation"]
    if cfg.samples > 1:
        parts.append(f"{st.num_seqs // cfg.samples} prompts x {cfg.samples} samples sharing "
                     f"ref-counted prompt blocks, prompt lengths {describe_lengths(cfg.lengths)}, "
                     f"divergent tails {describe_lengths(cfg.tail)} already cached (written before "
                     f"the timed steps, after {st.copy_pairs.shape[0]} copy-on-write block copies at "
                     f"divergence); each step writes every sample's newest K/V row "
                     f"({st.num_seqs} rows), then attends")
    else:
        parts.append(f"context lengths {describe_lengths(cfg.lengths)} "
                     f"(mean {st.context_lens.mean():.0f})")
        if st.num_new_tokens:
            parts.append(f"plus reshape_and_cache of {st.num_new_tokens} new rows")
    parts.append(f"{cfg.num_blocks}-block pools")
    parts.append(f"{attention} attention")
    if kv:
        parts.append(kv)
    return {
        "workload": ", ".join(parts),
        "global_batch": st.num_seqs * world,
        "seq_len": int(st.max_context_len),
        "parallelism": "single GPU" if world == 1 else f"{world} independent replicas",
        "l2": f"{flush_desc(flush)}; step inputs "
              f"{workload_bytes(st, 1 if kv else None, **step_counts(cfg, st))['step'] / 1e9:.2f} GB",
        "seed": cfg.seed,
    }


def peak_hbm() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback (6.8 TB/s)"


def peak_bf16_tflops() -> tuple[float, str]:
    """Dense bf16 tensor peak: the burst figure (the prefill kernel is timed
    alone between L2 flushes)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "of measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "of fallback (1.9 PFLOP/s bf16)"


def source_hash(files) -> str:
    """Hash of the kernel sources with their // comments and blank lines
    taken out, so that an edit of a comment keeps a recorded figure valid."""
    h = hashlib.sha256()
    for f in files:
        for line in open(os.path.join(CSRC, f), encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(kind: str = "plain") -> int | None:
    """DRAM bytes per launch of a kernel from its committed ncu summary, if
    the summary was taken on the current kernel sources."""
    path, files = PROFILES[kind]
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_traffic or m_hash.group(1) != source_hash(files):
        return None
    return int(m_traffic.group(1))


class ClockSampler:
    """SM clock, power and clock-event reasons of the GPU, polled from a
    background thread through NVML (read-only queries, by ctypes) every
    `period_s`; nvidia-smi polling when NVML cannot be loaded. Start it before
    the warm-up and call `mark_timed(t0, t1)` with the timed region's wall
    clock: the summary covers the samples inside it."""
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.device_index = device_index
        self.period = period_s
        self.samples: list[tuple[float, float, float, float, int]] = []  # (t, sm, max, watts, reasons)
        self.source = None
        self.window = None
        self._stop = None
        self._thread = None
        self._proc = None
        self._uuid = None
        try:
            import torch
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self._uuid = u if u.startswith("GPU-") else f"GPU-{u}"
        except Exception:
            pass

    # -- NVML ------------------------------------------------------------
    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        if self._uuid is None or lib.nvmlDeviceGetHandleByUUID(self._uuid.encode(), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle for the device")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        sm, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def read():
            lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm))      # NVML_CLOCK_SM
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            reasons_fn(h, ctypes.byref(rs))
            return float(sm.value), float(mx.value), mw.value / 1000.0, int(rs.value)
        read()
        return lib, read

    def _poll(self, read):
        while not self._stop.is_set():
            try:
                s = read()
            except Exception:
                break
            self.samples.append((time.perf_counter(), *s))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        try:
            self._lib, read = self._nvml()
            self.source = "nvml"
            self._thread = threading.Thread(target=self._poll, args=(read,), daemon=True)
            self._thread.start()
        except Exception:
            sel = ["-i", self._uuid] if self._uuid else []
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", *sel, f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self._t_smi = time.perf_counter()
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            try:
                self._lib.nvmlShutdown()
            except Exception:
                pass
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                out, _ = self._proc.communicate()
            lines = [l for l in out.splitlines() if l.strip()]
            t_end = time.perf_counter()
            names = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                     "sw_power_cap": 0x4}
            for k, line in enumerate(lines):  # spread evenly over the polling time (no timestamps)
                parts = [p.strip() for p in line.split(",")]
                try:
                    sm, mx = float(parts[0]), float(parts[1])
                    w = float(parts[2]) if parts[2].replace(".", "", 1).isdigit() else 0.0
                except (ValueError, IndexError):
                    continue
                bits = 0
                for (name, bit), val in zip(names.items(), parts[4:8]):
                    if val.lower() == "active":
                        bits |= bit
                t = self._t_smi + (t_end - self._t_smi) * (k + 0.5) / max(1, len(lines))
                self.samples.append((t, sm, mx, w, bits))

    def mark_timed(self, t0: float, t1: float) -> None:
        self.window = (t0, t1)

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source,
                    "note": "no clock samples"}
        sel, where = self.samples, "whole run (warm-up, timed region, end-to-end steps)"
        if self.window is not None:
            inside = [s for s in self.samples if self.window[0] <= s[0] <= self.window[1]]
            if inside:
                sel, where = inside, "timed region"
        reasons = sorted({name for s in sel for bit, name in self.REASON_BITS.items() if s[4] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": max(s[2] for s in sel),
                "sm_mhz_min": min(s[1] for s in sel), "power_w_max": max(s[3] for s in sel),
                "reasons": reasons, "samples": len(sel), "samples_total": len(self.samples),
                "window": where, "source": self.source}


class L2Flush:
    """Evicts the previous step's lines from L2 between timed steps: writes a
    buffer twice the L2's size and, in mode "write+read", then reads another
    buffer of that size, so that the written lines are back in HBM before
    the timed region starts and no write-back of the flush lands inside it."""

    def __init__(self, device, mode: str = "write+read"):
        import torch
        self.mode = mode
        self.wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64, device=device) if mode == "write+read" else None

    def __call__(self, i: int) -> None:
        self.wbuf.fill_(i & 0xFF)
        if self.rbuf is not None:
            self.rbuf.amax()

    def describe(self) -> str:
        return flush_desc(self.mode)

    @property
    def launches(self) -> int:
        return 2 if self.rbuf is not None else 1


def cpu_sample(cfg, n_seqs: int):
    """The first n_seqs sequences of the workload (same length draws), on the host."""
    import synth.host as H
    n_seqs = max(cfg.samples, min(n_seqs, cfg.num_seqs) // cfg.samples * cfg.samples)
    hw = H.generate(cfg, num_seqs=n_seqs)
    return hw, H.compact_pools(hw)


def time_oracle(cfg, min_seconds: float, n_seqs: int, max_runs: int | None = None) -> dict:
    """The fp64 oracle, as it stands, on the host cores: one step (new rows
    written, then attention) over a bounded sample of the workload, with one
    thread per core of the affinity mask and then with a single thread (on a
    quarter of the sample)."""
    import oracle
    import synth.host as H
    threads = len(os.sched_getaffinity(0))

    def timed(n, nthreads, seconds):
        hw, hp0 = cpu_sample(cfg, n)
        nbytes = workload_bytes(hw.st)["step"]
        times = []
        t_start = time.perf_counter()
        while True:
            hp = H.HostPools(hp0.k_cache.copy(), hp0.v_cache.copy(), hp0.block_tables, hp0.slot_mapping,
                             hp0.copy_pairs, hp0.ids, hp0.seqs, hp0.prefix_tables)
            t0 = time.perf_counter()
            oracle.decode_step(hp, hw, threads=nthreads)
            times.append(time.perf_counter() - t0)
            if time.perf_counter() - t_start >= seconds or (max_runs and len(times) >= max_runs):
                break
        mean = sum(times) / len(times)
        desc = (f"first {hw.st.num_seqs} of {cfg.num_seqs} sequences of the same workload "
                f"({int(hw.st.context_lens.sum())} tokens x {cfg.num_heads} heads), "
                f"{len(times)} run(s) of one step, {mean * 1e3:.1f} ms each")
        return nbytes / mean / 1e9, mean, nbytes, desc

    n_seqs = max(cfg.samples, min(n_seqs, cfg.num_seqs) // cfg.samples * cfg.samples)
    value, mean, nbytes, desc = timed(n_seqs, threads, min_seconds)
    n1 = max(cfg.samples, n_seqs // 4 // cfg.samples * cfg.samples)
    v1, _, _, desc1 = timed(n1, 1, min_seconds / 2)
    return {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
            "single_thread": {"value": v1, "unit": "GB/s", "cores": 1, "sample": desc1},
            "ms_per_step": mean * 1e3, "bytes_per_step": nbytes}


# ----------------------------------------------------------------- reference arm
def run_reference(args, rank: int, world: int) -> int:
    """The oracle as it stands on the host cores, on a bounded sample of the
    same workload per step: the first n sequences (n = cores, at most the
    batch) restricted to their first h heads, h sized so that warm-up plus
    the timed steps end within about two minutes."""
    if rank != 0:
        return 0
    import oracle
    import synth
    import synth.host as H
    cfg = synth.get(args.workload)
    st_full = synth.build(cfg)
    threads = len(os.sched_getaffinity(0))
    n = max(1, min(cfg.num_seqs, threads))

    def sample(h):
        c = cfg.replace(num_heads=h, num_kv_heads=h)
        return cpu_sample(c, n)

    def run(hw, hp0):
        hp = H.HostPools(hp0.k_cache.copy(), hp0.v_cache.copy(), hp0.block_tables, hp0.slot_mapping,
                         hp0.copy_pairs, hp0.ids, hp0.seqs, hp0.prefix_tables)
        t0 = time.perf_counter()
        oracle.decode_step(hp, hw, threads=threads)
        return time.perf_counter() - t0

    hw, hp0 = sample(1)
    per_head = run(hw, hp0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    h = int(max(1, min(cfg.num_heads, budget / max(per_head, 1e-6))))
    hw, hp0 = sample(h)
    nbytes = workload_bytes(hw.st)["step"]
    for _ in range(args.warmup):
        run(hw, hp0)
    times = [run(hw, hp0) for _ in range(args.steps)]
    mean = sum(times) / len(times)
    value = nbytes / mean / 1e9
    sample_desc = (f"first {n} of {cfg.num_seqs} sequences x first {h} of {cfg.num_heads} heads per step "
                   f"({int(hw.st.context_lens.sum())} tokens)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_json(cfg, st_full, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm
def pack_inputs(tensors, dev):
    """One device buffer holding every tensor (each at a 256-byte aligned
    offset, filled with its current contents), the views of it that replace
    the tensors, and a pinned host buffer with the same bytes: a step's inputs
    then travel in one host-to-device copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    dbuf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        v = dbuf[o:o + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    hbuf = dbuf.cpu().pin_memory()
    return dbuf, hbuf, views


def aggregate(values: dict, world: int, device=None) -> dict:
    """Max of each timing over ranks (identity for one rank)."""
    if world == 1:
        return dict(values)
    import torch
    import torch.distributed as dist
    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {k: float(v) for k, v in zip(keys, t.tolist())}


# fp8 pools: one scale per pool; |x| up to 6 (6 sigma of the N(0, 1) values) maps to 448
FP8_SCALE = 6.0 / 448.0


def fp8_pool(pool, scale: float, chunk: int = 2048):
    """A 16-bit pool as e4m3 codes (uint8, same shape): x / scale clamped to
    +-448 and rounded by PyTorch's float8 conversion; poisoned (NaN) rows stay
    NaN. Input generation only: the timed step writes its rows with the
    library's fp8 cache write."""
    import torch
    out = torch.empty(pool.shape, dtype=torch.uint8, device=pool.device)
    for a in range(0, pool.shape[0], chunk):
        x = (pool[a:a + chunk].float() / scale).clamp_(-448.0, 448.0)
        out[a:a + chunk] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def q4_pool(pool, scale_sigma: float, seed: int, chunk: int = 2048):
    """q4_0 rows (uint8 [blocks, kv heads, block_size, 9 D / 16]) in place of
    a 16-bit pool: uniform random code bytes and binary16 scales drawn from
    N(0, scale_sigma^2), values of the same spread as the 16-bit data. Input
    generation only: the timed step writes its rows with the library's q4_0
    cache write."""
    import torch
    nb, hkv, bs, d = pool.shape
    rb = d // 16 * 9
    out = torch.empty((nb, hkv, bs, rb), dtype=torch.uint8, device=pool.device)
    gen = torch.Generator(device=pool.device)
    gen.manual_seed(seed)
    for a in range(0, nb, chunk):
        o = out[a:a + chunk]
        o.copy_(torch.randint(0, 256, o.shape, generator=gen, device=pool.device, dtype=torch.int32).to(torch.uint8))
        sc = (torch.randn(o.shape[:3] + (d // 32,), generator=gen, device=pool.device) * scale_sigma).half()
        o[..., :d // 16] = sc.view(torch.uint8)
    return out


def kv_memory(cfg) -> dict:
    """KV memory of the workload as the library's host block manager lays it
    out ("PagedAttention: the KV cache was the bottleneck all along", sections
    "Virtual memory for attention" and "The number that made us read the
    code"), and the host time of one decode step's bookkeeping (one more slot
    for every sequence, then the block tables and context lengths)."""
    import paged_kv_cache_204_gb300.block_manager as pbm
    from synth.replay import replay

    m = pbm.BlockManager(cfg.num_blocks, cfg.block_size, seed=cfg.seed)
    seqs = replay(m, cfg)
    st = m.stats()
    mm = pbm.memory_metrics(st, cfg.block_size)
    ones = [1] * len(seqs)
    reps = 50
    t0 = time.perf_counter()
    for _ in range(reps):
        m.append_batch(seqs, ones)
        m.export(seqs, cfg.max_blocks_per_seq + reps)
    step_us = (time.perf_counter() - t0) / reps * 1e6
    return {"waste_fraction": mm["waste_fraction"], "sharing_saving": mm["sharing_saving"],
            "contiguous_reservation_waste": 1.0 - st["logical_tokens"] / (st["live_seqs"] * cfg.max_len),
            "reserved_tokens_per_sequence": cfg.max_len,
            "used_blocks": st["used_blocks"], "logical_blocks": st["logical_blocks"],
            "cow_copies": st["cow_copies"], "host_step_us": step_us}


def run_ours(args, rank: int, world: int, local_rank: int) -> int:
    import torch
    import torch.distributed as dist

    import paged_kv_cache_204_gb300 as pkv
    import synth
    import synth.device as SD

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    cfg = synth.get(args.workload)
    if args.num_blocks:
        cfg = cfg.replace(num_blocks=args.num_blocks)
    if world > 1:
        cfg = cfg.replace(seed=cfg.seed + rank)
    dw = SD.generate(cfg, device=dev)
    st = dw.st
    cow = cfg.samples > 1
    cow_copy_us = None
    if cow:
        # Copy-on-write history: the copies at divergence and the samples'
        # tails are written once here (copy_blocks timed on its own); a timed
        # step then writes each sample's newest row (its last tail token,
        # the same values again) and attends.
        err0 = torch.zeros(1, dtype=torch.int32, device=dev)
        flush0 = L2Flush(dev, args.flush)
        copy_times = []
        for i in range(8):  # the copies, then the tails (which rewrite the copied blocks' tail rows)
            flush0(i)
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record()
            pkv.copy_blocks(dw.k_cache, dw.v_cache, dw.copy_pairs, dev_err=err0)
            c1.record()
            pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=err0)
            torch.cuda.synchronize()
            copy_times.append(c0.elapsed_time(c1) * 1e3)
        del flush0
        if int(err0.item()) != 0:
            raise RuntimeError(f"device error word {int(err0.item()):#x} while writing the tails")
        cow_copy_us = statistics.median(copy_times[3:])  # warm launches, L2 flushed before each
        last = torch.from_numpy(st.new_start[1:] - 1).to(dev)
        dw.new_k, dw.new_v = dw.new_k[last].contiguous(), dw.new_v[last].contiguous()
        dw.slot_mapping = dw.slot_mapping[last].contiguous()
        dw.copy_pairs = dw.copy_pairs[:0]
    fp8, q4 = args.kv == "fp8", args.kv == "q4_0"
    if (fp8 or q4) and (args.attention != "plain" or cfg.dtype == "f32"):
        raise SystemExit(f"--kv {args.kv} takes the plain attention of a 16-bit workload")
    if fp8:
        dw.k_cache = fp8_pool(dw.k_cache, FP8_SCALE)
        dw.v_cache = fp8_pool(dw.v_cache, FP8_SCALE)
        torch.cuda.empty_cache()
    if q4:
        # a 32-value block of N(0, s^2) values spans about 3 s: scales near 3 s / 8
        dw.k_cache = q4_pool(dw.k_cache, 0.4 * cfg.value_scale, cfg.seed + 1)
        dw.v_cache = q4_pool(dw.v_cache, 0.4 * cfg.value_scale, cfg.seed + 2)
        torch.cuda.empty_cache()
    kv_desc = (f"fp8 e4m3 K/V pools (per-pool scale {FP8_SCALE:.6g}; new rows rounded on write)" if fp8 else
               f"q4_0 K/V pools (blocks of 32 values, binary16 scale, 4-bit codes; {cfg.head_dim // 16 * 9}-byte "
               f"rows; new rows quantised on write)" if q4 else None)
    nbytes = workload_bytes(st, 1 if fp8 else None, new_rows=int(dw.slot_mapping.numel()),
                            copy_pairs=int(dw.copy_pairs.shape[0]),
                            kv_row_bytes=cfg.head_dim // 16 * 9 if q4 else None)
    B, H, D = st.num_seqs, cfg.num_heads, cfg.head_dim
    mcl = st.max_context_len
    grouped = args.attention == "grouped"
    if grouped and st.group_start is None:
        raise SystemExit(f"--attention grouped needs a workload with sharing groups, not {cfg.name}")
    if grouped:
        gs = torch.from_numpy(st.group_start).to(dev)
        sb = torch.from_numpy(st.shared_blocks).to(dev)
        ws = pkv.new_grouped_workspace(B, H, D, mcl, sb.numel(), device=dev)
    else:
        ws = pkv.new_workspace(B, H, D, mcl, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(dw.q)
    flush = L2Flush(dev, args.flush)
    stream = torch.cuda.current_stream(dev)
    has_copy, has_new = dw.copy_pairs.numel() > 0, dw.slot_mapping.numel() > 0

    def cache_ops():
        if has_copy:
            pkv.copy_blocks(dw.k_cache, dw.v_cache, dw.copy_pairs, dev_err=err)
        if has_new:
            if fp8:
                pkv.reshape_and_cache_fp8(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, FP8_SCALE,
                                          FP8_SCALE, dev_err=err)
            elif q4:
                pkv.reshape_and_cache_q4_0(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=err)
            else:
                pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=err)

    def attention():
        if fp8:
            pkv.paged_attention_decode_fp8(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                                           cfg.scale, FP8_SCALE, FP8_SCALE, mcl, workspace=ws, dev_err=err)
        elif q4:
            pkv.paged_attention_decode_q4_0(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                                            cfg.scale, mcl, workspace=ws, dev_err=err)
        elif grouped:
            pkv.paged_attention_decode_grouped(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                               dw.context_lens, cfg.scale, mcl, gs, sb, ws, dev_err=err)
        else:
            pkv.paged_attention_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                       dw.context_lens, cfg.scale, mcl, workspace=ws, dev_err=err)

    def step():
        cache_ops()
        attention()

    # grouped: the grouping check, then one kernel (16-bit data) or a prefix and a tail phase (fp32)
    launches_per_step = int(has_copy) + int(has_new) + ((3 if cfg.dtype == "f32" else 2) if grouped else 1)

    clocks = ClockSampler(local_rank).__enter__()  # sampled from the warm-up on
    for _ in range(max(args.warmup, 3)):
        flush(1)
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} during warm-up")
    if not torch.isfinite(out.float()).all():
        raise RuntimeError("non-finite output during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush(i)  # evict the previous step's lines from L2
        ev[i][0].record(stream)
        cache_ops()
        ev[i][1].record(stream)
        attention()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clocks.mark_timed(t_wall0, t_wall0 + wall)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    decode_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    cache_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} in the timed region")

    # end to end through the same API with host buffers: per step, copy the
    # step's inputs from pinned host memory (packed: one copy), run the step,
    # read the output back
    names = [n for n in ("q", "new_k", "new_v", "slot_mapping", "block_tables", "context_lens", "copy_pairs")
             if getattr(dw, n).numel()]
    dev_in = [getattr(dw, n) for n in names] + ([gs, sb] if grouped else [])
    dbuf, hbuf, views = pack_inputs(dev_in, dev)
    for n, v in zip(names, views):
        setattr(dw, n, v)
    if grouped:
        gs, sb = views[-2:]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = hbuf.numel()
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(10, K // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_total = 0.0
    for i in range(e2e_steps + 3):
        flush(i)
        if i >= 3:
            e0.record(stream)
        dbuf.copy_(hbuf, non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        if i >= 3:
            e1.record(stream)
            e1.synchronize()
            e2e_total += e0.elapsed_time(e1)
    e2e_ms = e2e_total / e2e_steps
    clocks.__exit__(None, None, None)

    agg = aggregate({"step_ms": step_ms, "decode_ms": decode_ms, "cache_ms": cache_ms, "e2e_ms": e2e_ms},
                    world, device=dev if world > 1 else None)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_src = peak_hbm()
    achieved = nbytes["attention"] / (agg["decode_ms"] * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        if fp8:
            cpu = sampled_attention_baseline(cfg, dw.k_cache, dw.v_cache, st.block_tables, st.context_lens, dw.q,
                                             args.cpu_seconds, args.cpu_seqs, "sequences (fp8 pools)",
                                             fp8_scales=(FP8_SCALE, FP8_SCALE))
        elif q4:
            cpu = sampled_attention_baseline(cfg, dw.k_cache, dw.v_cache, st.block_tables, st.context_lens, dw.q,
                                             args.cpu_seconds, args.cpu_seqs, "sequences (q4_0 pools)", q4=True)
        elif cow:
            cpu = sampled_attention_baseline(cfg, dw.k_cache, dw.v_cache, st.block_tables, st.context_lens, dw.q,
                                             args.cpu_seconds, args.cpu_seqs, "samples (plain paged attention)")
        else:
            cpu = time_oracle(cfg, args.cpu_seconds, args.cpu_seqs)
            cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "single_thread")}
    line = {
        "metric": METRIC,
        "value": world * nbytes["step"] / (agg["step_ms"] * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": agg["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"{cfg.dtype} queries, fp8_e4m3 K/V" if fp8 else f"{cfg.dtype} queries, q4_0 K/V" if q4
                  else cfg.dtype), "data": "synthetic",
        "config": config_json(cfg, st, world, args.attention, kv_desc, args.flush),
        "seqs_per_s": world * B / (agg["step_ms"] * 1e-3),
        "attention_ms": agg["decode_ms"], "cache_ops_ms": agg["cache_ms"],
        "bytes_per_step": nbytes["step"], "roofline_frac_step": nbytes["step"] / (agg["step_ms"] * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm",
                     "kernel": ("pa_group_prologue + pa_decode_shared_kernel" if grouped else
                                "pa_decode_kernel<fp8 e4m3 cache>" if fp8 else
                                "pa_decode_kernel<q4_0 cache>" if q4 else "pa_decode_kernel"),
                     "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": (profiled_traffic("fp8") if fp8 else profiled_traffic("q4") if q4 else
                                 profiled_traffic("plain"))
                     if (cfg.name == WORKLOAD and not grouped) else
                     profiled_traffic("grouped") if (cfg.name == "cow" and grouped) else None,
                     "algorithmic_bytes_per_launch": nbytes["attention"], "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": world * nbytes["step"] / (agg["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": agg["e2e_ms"], "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        **({"cow_copy_blocks_us": cow_copy_us, "cow_copy_pairs": int(st.copy_pairs.shape[0])} if cow else {}),
        "clocks": clocks.summary(),
        "timed_region_wall_s": wall,
        "kv_memory": kv_memory(cfg),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def sampled_attention_baseline(cfg, kc, vc, block_tables, context_lens, q, min_seconds: float, n_seqs: int,
                               what: str, fp8_scales=None, q4: bool = False) -> dict:
    """The fp64 oracle, as it stands, on the host cores: paged attention of
    the first n_seqs sequences over host copies of their blocks (fp8 pools
    when fp8_scales = (k_scale, v_scale), q4_0 pools when q4), repeated for
    about min_seconds."""
    import numpy as np
    import oracle
    from synth.device import to_storage
    threads = len(os.sched_getaffinity(0))
    n = max(1, min(n_seqs, len(context_lens)))
    bt, cl = np.ascontiguousarray(block_tables[:n]), np.ascontiguousarray(context_lens[:n])
    ids = np.unique(bt[bt >= 0])
    remap = np.full(cfg.num_blocks, -1, dtype=np.int32)
    remap[ids] = np.arange(ids.size, dtype=np.int32)
    bt_c = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    import torch
    idx = torch.from_numpy(ids.astype(np.int64)).to(kc.device)
    q_h = to_storage(q[:n])
    if fp8_scales is None and not q4:
        k_h, v_h = to_storage(kc[idx]), to_storage(vc[idx])
    else:
        k_h, v_h = kc[idx].cpu().numpy(), vc[idx].cpu().numpy()
    rows = {(int(b), r) for i in range(n) for j, b in enumerate(bt[i][bt[i] >= 0])
            for r in range(min(cfg.block_size, int(cl[i]) - j * cfg.block_size))}
    kv_row = (2 * cfg.num_kv_heads * (cfg.head_dim // 16 * 9) if q4 else
              cfg.kv_bytes_per_token() // (1 if fp8_scales is None else cfg.elem_bytes))
    nbytes = len(rows) * kv_row + 2 * n * cfg.num_heads * cfg.head_dim * cfg.elem_bytes
    kw = dict(num_heads=cfg.num_heads, num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim,
              block_size=cfg.block_size, threads=threads)
    times, t_start = [], time.perf_counter()
    while True:
        t0 = time.perf_counter()
        if q4:
            oracle.paged_attention_q4_0(q_h, k_h, v_h, bt_c, cl, scale=cfg.scale, q_dtype=cfg.dtype, **kw)
        elif fp8_scales is None:
            oracle.paged_attention(q_h, k_h, v_h, bt_c, cl, scale=cfg.scale, dtype=cfg.dtype, **kw)
        else:
            oracle.paged_attention_fp8(q_h, k_h, v_h, bt_c, cl, scale=cfg.scale, k_scale=fp8_scales[0],
                                       v_scale=fp8_scales[1], q_dtype=cfg.dtype, **kw)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= min_seconds:
            break
    mean = sum(times) / len(times)
    return {"value": nbytes / mean / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"attention of the first {n} of {len(context_lens)} {what} "
                       f"({int(cl.sum())} tokens x {cfg.num_heads} heads, {len(rows)} distinct cached tokens), "
                       f"{len(times)} run(s), {mean * 1e3:.1f} ms each")}


def run_beam(args, rank: int, world: int, local_rank: int) -> int:
    """Beam-search decode steps: per step the block manager forks and ends
    beams, copy_blocks copies shared partly filled blocks, reshape_and_cache
    writes every new beam's K/V row, and the grouped decode reads each
    request's shared prefix once for all its beams. The timed region runs the
    device part of each step with that step's plan (block tables, slots,
    copy pairs, groups) already resident; e2e runs further steps through
    BeamDecoder.step, host bookkeeping and transfers included."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_kv_cache_204_gb300 as pkv
    import synth.beam as SB
    from paged_kv_cache_204_gb300.beam import BeamDecoder, DevicePlan
    from synth.device import fill_poison

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    warm = max(args.warmup, 3)
    K = args.steps
    e2e_steps = max(10, K // 4)
    cfg = SB.get(args.workload)
    cfg = cfg.replace(steps=max(cfg.steps, warm + K + e2e_steps + 3))
    if args.num_blocks:
        cfg = cfg.replace(num_blocks=args.num_blocks)
    if world > 1:
        cfg = cfg.replace(seed=cfg.seed + rank)
    td = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[cfg.dtype]
    shape = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    kc = torch.empty(shape, dtype=td, device=dev)
    vc = torch.empty(shape, dtype=td, device=dev)
    fill_poison(kc)
    fill_poison(vc)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed * 1000003 + 29)
    randn = lambda *shp: (torch.randn(shp, generator=gen, device=dev) * cfg.value_scale).to(td)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dec = BeamDecoder(kc, vc, cfg.width, cfg.max_blocks_per_seq, seed=cfg.seed)
    for P in SB.prompt_lengths(cfg):
        dec.add_request(randn(int(P), cfg.num_kv_heads, cfg.head_dim), randn(int(P), cfg.num_kv_heads, cfg.head_dim),
                        dev_err=err)
    B, H, D = cfg.num_seqs, cfg.num_heads, cfg.head_dim
    nk, nv, q = randn(B, cfg.num_kv_heads, D), randn(B, cfg.num_kv_heads, D), randn(B, H, D)
    out = torch.empty_like(q)
    parents_of = SB.parent_stream(cfg)
    row_bytes = cfg.kv_bytes_per_token()
    block_bytes = row_bytes * cfg.block_size
    dplans, step_bytes, attn_bytes, n_copies = [], [], [], 0
    for i in range(warm + K):
        plan = dec.plan(next(parents_of))
        st = dec.manager.stats()  # the live sequences are exactly the beams
        a_bytes = st["filled_slots"] * row_bytes + 2 * B * H * D * cfg.elem_bytes
        c = plan.copy_pairs.shape[0]
        n_copies += c
        attn_bytes.append(a_bytes)
        step_bytes.append(a_bytes + 2 * B * row_bytes + 2 * c * block_bytes)
        dplans.append(DevicePlan(max_context_len=plan.max_context_len, **{
            name: torch.from_numpy(np.ascontiguousarray(getattr(plan, name))).to(dev)
            for name in ("slots", "copy_pairs", "block_tables", "context_lens", "group_start", "shared_blocks")}))
    ws = dec.workspace(H, D)
    flush = L2Flush(dev, args.flush)
    stream = torch.cuda.current_stream(dev)

    def device_step(dp, e_write=None):
        if dp.copy_pairs.numel():
            pkv.copy_blocks(kc, vc, dp.copy_pairs, dev_err=err)
        pkv.reshape_and_cache(nk, nv, kc, vc, dp.slots, dev_err=err)
        if e_write is not None:  # copies and row writes done
            e_write.record(stream)
        pkv.paged_attention_decode_grouped(out, q, kc, vc, dp.block_tables, dp.context_lens, cfg.scale,
                                           dp.max_context_len, dp.group_start, dp.shared_blocks, ws, dev_err=err)

    clocks = ClockSampler(local_rank).__enter__()  # sampled from the warm-up on
    for i in range(warm):
        flush(1)
        device_step(dplans[i])
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    t_wall0 = time.perf_counter()
    for i in range(K):
        dp = dplans[warm + i]
        flush(i)
        ev[i][0].record(stream)
        device_step(dp, ev[i][1])
        ev[i][2].record(stream)
        # copies, the row writes, the grouping check and the grouped kernel (16-bit data) or its
        # prefix and tail phases (fp32)
        launches += (1 if dp.copy_pairs.numel() else 0) + 1 + (3 if cfg.dtype == "f32" else 2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clocks.mark_timed(t_wall0, t_wall0 + wall)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} in the timed region")
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    cache_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    bytes_step = sum(step_bytes[warm:]) / K
    bytes_attn = sum(attn_bytes[warm:]) / K

    # end to end: host bookkeeping, transfers of the plan and of q / new rows
    # from pinned host memory, the device step, and the outputs read back
    host_k, host_v, host_q = nk.cpu().pin_memory(), nv.cpu().pin_memory(), q.cpu().pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_total, h2d = 0.0, 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = 0
    for i in range(e2e_steps + 3):
        flush(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        plan = dec.plan(next(parents_of))
        dp = dec.upload(plan)
        nk.copy_(host_k, non_blocking=True)
        nv.copy_(host_v, non_blocking=True)
        q.copy_(host_q, non_blocking=True)
        dec.run(dp, nk, nv, q, cfg.scale, out, dev_err=err)
        host_out.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        if i >= 3:
            e2e_total += time.perf_counter() - t0
            st = dec.manager.stats()
            e2e_bytes += (st["filled_slots"] * row_bytes + 2 * B * H * D * cfg.elem_bytes + 2 * B * row_bytes
                          + 2 * plan.copy_pairs.shape[0] * block_bytes)
            h2d += sum(getattr(plan, f).nbytes for f in ("slots", "copy_pairs", "block_tables", "context_lens",
                                                         "group_start", "shared_blocks"))
            h2d += sum(t.numel() * t.element_size() for t in (host_k, host_v, host_q))
    e2e_ms = e2e_total / e2e_steps * 1e3
    clocks.__exit__(None, None, None)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} in the end-to-end steps")

    agg = aggregate({"step_ms": step_ms, "attn_ms": attn_ms, "cache_ms": cache_ms, "e2e_ms": e2e_ms},
                    world, device=dev if world > 1 else None)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_src = peak_hbm()
    achieved = bytes_attn / (agg["attn_ms"] * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        cpu = sampled_attention_baseline(cfg, kc, vc, plan.block_tables, plan.context_lens, q, args.cpu_seconds,
                                         args.cpu_seqs, "beams at the last step")
    st = dec.manager.stats()
    import paged_kv_cache_204_gb300.block_manager as pbm
    mm = pbm.memory_metrics(st, cfg.block_size)
    line = {
        "metric": METRIC,
        "value": world * bytes_step / (agg["step_ms"] * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": warm,
        "ms_per_step": agg["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": (f"beam-search decode steps: {cfg.requests} requests x {cfg.width} beams, "
                                f"{H} heads ({cfg.num_kv_heads} kv), head_dim {D}, block_size {cfg.block_size}, "
                                f"{cfg.dtype} storage with fp32 accumulation, prompts {cfg.prompt[0]} in "
                                f"[{cfg.prompt[1]}, {cfg.prompt[2]}], parents drawn with rank weights (W-j)^2, "
                                f"{cfg.num_blocks}-block pools, grouped attention (one group per request)"),
                   "global_batch": B, "parallelism": "single GPU" if world == 1 else f"{world} replicas",
                   "l2": flush.describe(), "seed": cfg.seed,
                   "copies_per_step": n_copies / (warm + K)},
        "seqs_per_s": world * B / (agg["step_ms"] * 1e-3),
        "attention_ms": agg["attn_ms"], "cache_ops_ms": agg["cache_ms"],
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "kernel": "pa_group_prologue + pa_decode_shared_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "algorithmic_bytes_per_launch": bytes_attn, "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": world * (e2e_bytes / e2e_steps) / (agg["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": agg["e2e_ms"], "h2d_bytes_per_step": h2d // e2e_steps,
                "d2h_bytes_per_step": host_out.numel() * host_out.element_size()},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "timed_region_wall_s": wall,
        "kv_memory": {"waste_fraction": mm["waste_fraction"], "sharing_saving": mm["sharing_saving"],
                      "used_blocks": st["used_blocks"], "logical_blocks": st["logical_blocks"],
                      "cow_copies": st["cow_copies"]},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_prefill(args, rank: int, world: int, local_rank: int) -> int:
    """Prefill steps of users sharing a system prompt: the system prompt's
    K/V is in the cache already (written once, its partly filled block copied
    on write for the users); each step writes the users' own K/V rows and
    runs the causal prefill attention of all their tokens."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_kv_cache_204_gb300 as pkv
    import synth.prefill as SP

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    cfg = SP.get(args.workload)
    if args.num_blocks:
        cfg = cfg.replace(num_blocks=args.num_blocks)
    if world > 1:
        cfg = cfg.replace(seed=cfg.seed + rank)
    lay = SP.build(cfg)
    td = {"f16": torch.float16, "bf16": torch.bfloat16}[cfg.dtype]
    H, Hkv, D = cfg.num_heads, cfg.num_kv_heads, cfg.head_dim
    n = lay.total_queries
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed * 1000003 + 31)
    randn = lambda *shp: (torch.randn(shp, generator=gen, device=dev) * cfg.value_scale).to(td)
    shape = (cfg.num_blocks, Hkv, cfg.block_size, D)
    kc = torch.full(shape, float("nan"), dtype=td, device=dev)
    vc = torch.full(shape, float("nan"), dtype=td, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if cfg.system_len:
        pkv.reshape_and_cache(randn(cfg.system_len, Hkv, D), randn(cfg.system_len, Hkv, D), kc, vc,
                              t(lay.system_slots), dev_err=err)
    if lay.copy_pairs.size:
        pkv.copy_blocks(kc, vc, t(lay.copy_pairs), dev_err=err)
    uk, uv, q = randn(n, Hkv, D), randn(n, Hkv, D), randn(n, H, D)
    slots, bt, cl, qs = t(lay.user_slots), t(lay.block_tables), t(lay.context_lens), t(lay.query_start)
    out = torch.empty_like(q)
    flush = L2Flush(dev, args.flush)
    stream = torch.cuda.current_stream(dev)

    def write():
        pkv.reshape_and_cache(uk, uv, kc, vc, slots, dev_err=err)

    def attention():
        pkv.paged_attention_prefill(out, q, kc, vc, bt, cl, qs, cfg.scale, lay.max_query_len, dev_err=err)

    # algorithmic work: every query sees the system prompt and its own earlier tokens
    visible = 0
    for u in range(cfg.users):
        nu = int(lay.query_start[u + 1] - lay.query_start[u])
        L = int(lay.context_lens[u])
        visible += sum(L - nu + i + 1 for i in range(nu))
    flops = 4.0 * visible * H * D
    warm = max(args.warmup, 3)
    clocks = ClockSampler(local_rank).__enter__()  # sampled from the warm-up on
    for _ in range(warm):
        flush(1)
        write()
        attention()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} during warm-up")
    if not torch.isfinite(out.float()).all():
        raise RuntimeError("non-finite prefill output")
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        write()
        ev[i][1].record(stream)
        attention()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clocks.mark_timed(t_wall0, t_wall0 + wall)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} in the timed region")
    # end to end: the users' rows, queries and layout from pinned host memory,
    # the step, the outputs back
    dbuf, hbuf, views = pack_inputs([uk, uv, q, slots, bt, cl, qs], dev)
    uk, uv, q, slots, bt, cl, qs = views
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps, e2e_total = max(10, K // 4), 0.0
    for i in range(e2e_steps + 3):
        flush(i)
        if i >= 3:
            e0.record(stream)
        dbuf.copy_(hbuf, non_blocking=True)
        write()
        attention()
        host_out.copy_(out, non_blocking=True)
        if i >= 3:
            e1.record(stream)
            e1.synchronize()
            e2e_total += e0.elapsed_time(e1)
    e2e_ms = e2e_total / e2e_steps
    clocks.__exit__(None, None, None)
    agg = aggregate({"step_ms": step_ms, "attn_ms": attn_ms, "write_ms": write_ms, "e2e_ms": e2e_ms}, world,
                    device=dev if world > 1 else None)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_src = peak_bf16_tflops()
    achieved = flops / (agg["attn_ms"] * 1e-3) / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        from synth.device import to_storage
        threads = len(os.sched_getaffinity(0))
        u = 0
        ids = np.unique(lay.block_tables[u][lay.block_tables[u] >= 0])
        remap = np.full(cfg.num_blocks, -1, dtype=np.int32)
        remap[ids] = np.arange(ids.size, dtype=np.int32)
        bt_c = np.where(lay.block_tables[u:u + 1] >= 0, remap[np.maximum(lay.block_tables[u:u + 1], 0)], -1)
        idx = torch.from_numpy(ids.astype(np.int64)).to(dev)
        nu = int(lay.query_start[1])
        hk = max(1, min(H, 2))  # a bounded sample: the first user's queries, first heads
        q_h = to_storage(q[:nu, :hk].contiguous())
        k_h = to_storage(kc[idx][:, :hk].contiguous()) if Hkv == H else to_storage(kc[idx])
        v_h = to_storage(vc[idx][:, :hk].contiguous()) if Hkv == H else to_storage(vc[idx])
        hkv = hk if Hkv == H else Hkv
        L0 = int(lay.context_lens[0])
        fl = 4.0 * sum(L0 - nu + i + 1 for i in range(nu)) * hk * D
        times, t_start = [], time.perf_counter()
        while True:
            t0 = time.perf_counter()
            oracle.paged_prefill(q_h, k_h, v_h, bt_c.astype(np.int32), lay.context_lens[:1],
                                 np.array([0, nu], dtype=np.int32), scale=cfg.scale, num_heads=hk,
                                 num_kv_heads=hkv, head_dim=D, block_size=cfg.block_size, dtype=cfg.dtype,
                                 threads=threads)
            times.append(time.perf_counter() - t0)
            if time.perf_counter() - t_start >= args.cpu_seconds:
                break
        mean = sum(times) / len(times)
        cpu = {"value": fl / mean / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": (f"prefill of user 0 ({nu} queries over {L0} tokens) x {hk} of {H} heads, "
                          f"{len(times)} run(s), {mean * 1e3:.1f} ms each; the oracle runs one thread per sequence")}
    line = {
        "metric": "prefill attention TFLOP/s (causal, users sharing a system prompt)",
        "value": world * flops / (agg["step_ms"] * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": warm, "ms_per_step": agg["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": (f"prefill step: {cfg.users} users sharing a {cfg.system_len}-token system prompt "
                                f"(its blocks shared, {lay.copy_pairs.shape[0]} copy-on-write copies), own prompts "
                                f"{describe_lengths(cfg.user_len)} ({n} query tokens), {H} heads ({Hkv} kv), "
                                f"head_dim {D}, block_size {cfg.block_size}, {cfg.dtype} with fp32 accumulation, "
                                f"{cfg.num_blocks}-block pools"),
                   "global_batch": n * world, "parallelism": "single GPU" if world == 1 else f"{world} replicas",
                   "l2": flush.describe(), "seed": cfg.seed},
        "tokens_per_s": world * n / (agg["step_ms"] * 1e-3),
        "attention_ms": agg["attn_ms"], "cache_write_ms": agg["write_ms"], "flops_per_step": flops,
        "roofline": {"bound": "tensor", "kernel": "pa_prefill_kernel (tcgen05.mma, TMEM accumulators, TMA-fed K/V)", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (agg["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": agg["e2e_ms"],
                "h2d_bytes_per_step": hbuf.numel(),
                "d2h_bytes_per_step": host_out.numel() * host_out.element_size()},
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
        "timed_region_wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="synthetic workload preset (default: the LLaMA-13B-shaped step); "
                         "'beam': beam-search decode steps")
    ap.add_argument("--kv", choices=("native", "fp8", "q4_0"), default="native",
                    help="fp8: K/V pools of e4m3 codes with one scale per pool; q4_0: 4-bit blocks of 32 values "
                         "with a binary16 scale (plain attention)")
    ap.add_argument("--attention", choices=("plain", "grouped"), default="plain",
                    help="grouped: siblings read shared prefix blocks once (copy-on-write workloads)")
    ap.add_argument("--flush", choices=("write+read", "write"), default="write+read",
                    help="L2 flush between timed steps: write 256 MiB and then read another 256 MiB "
                         "(default), or only write (its dirty lines are then written back inside the "
                         "next timed kernel)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="minimum time of the CPU baseline")
    ap.add_argument("--cpu-seqs", type=int, default=32, help="sequences in the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-blocks", type=int, default=0,
                    help="physical blocks per pool (default: the workload's 40000); the same "
                         "sequences and K/V bytes in a smaller pool, for profiler captures")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.workload.startswith("prefill"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the default workload"}))
            return 0
        return run_prefill(args, rank, world, local_rank)
    if args.workload.startswith("beam"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the default workload"}))
            return 0
        return run_beam(args, rank, world, local_rank)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
