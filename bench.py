#!/usr/bin/env python
"""Benchmark of the paged decode hot path on the LLaMA-13B-shaped workload.

One step = one layer's decode step of the workload: reshape_and_cache of the
128 new K/V rows into their cache slots, then paged decode attention of the
128 query tokens (40 heads, head_dim 128, bf16) over their 16..2048-token
contexts scattered through a 40 000-block pool. Inputs are seeded synthetic
data resident in HBM; L2 is flushed (256 MiB write) between timed steps and
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
PROFILE = os.path.join(ROOT, "profiles", "pa_decode_llama13b.md")
DECODE_SOURCE = os.path.join(ROOT, "paged_kv_cache_204_gb300", "csrc", "decode.cuh")
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def workload_bytes(st) -> dict:
    """Algorithmic bytes of one step: attention reads each distinct cached
    (block, row) once for K and once for V plus q, and writes out; the cache
    write reads the new rows and writes them into the pools; each
    copy-on-write pair reads and writes one whole block of both pools."""
    cfg = st.cfg
    es = cfg.elem_bytes
    row = cfg.num_kv_heads * cfg.head_dim * es           # one token, one of K/V, all kv heads
    qo = st.num_seqs * cfg.num_heads * cfg.head_dim * es
    attn = 2 * st.unique_kv_tokens() * row + 2 * qo
    cache_write = 2 * 2 * st.num_new_tokens * row
    copies = 2 * 2 * st.copy_pairs.shape[0] * cfg.block_size * row
    return {"attention": attn, "cache_write": cache_write, "copy": copies,
            "step": attn + cache_write + copies}


def describe_lengths(spec) -> str:
    if spec[0] == "lognormal":
        return f"lognormal(median {spec[1]}, sigma {spec[2]}) clipped to [{spec[3]}, {spec[4]}]"
    if spec[0] == "uniform":
        return f"uniform in [{spec[1]}, {spec[2]}]"
    return f"fixed {list(spec[1])}"


def config_json(cfg, st, world: int, attention: str = "plain") -> dict:
    parts = [f"{cfg.name}-shaped decode step: {st.num_seqs} seqs, {cfg.num_heads} heads "
             f"({cfg.num_kv_heads} kv), head_dim {cfg.head_dim}, block_size {cfg.block_size}, "
             f"{cfg.dtype} storage with fp32 accumulation"]
    if cfg.samples > 1:
        parts.append(f"{st.num_seqs // cfg.samples} prompts x {cfg.samples} samples sharing "
                     f"ref-counted prompt blocks, prompt lengths {describe_lengths(cfg.lengths)}, "
                     f"divergent tails {describe_lengths(cfg.tail)}, {st.copy_pairs.shape[0]} "
                     f"copy-on-write block copies and {st.num_new_tokens} tail rows written per step")
    else:
        parts.append(f"context lengths {describe_lengths(cfg.lengths)} "
                     f"(mean {st.context_lens.mean():.0f})")
        if st.num_new_tokens:
            parts.append(f"plus reshape_and_cache of {st.num_new_tokens} new rows")
    parts.append(f"{cfg.num_blocks}-block pools")
    parts.append(f"{attention} attention")
    return {
        "workload": ", ".join(parts),
        "global_batch": st.num_seqs * world,
        "seq_len": int(st.max_context_len),
        "parallelism": "single GPU" if world == 1 else f"{world} independent replicas",
        "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB write); step inputs "
              f"{workload_bytes(st)['step'] / 1e9:.2f} GB",
        "seed": cfg.seed,
    }


def peak_hbm() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback (6.8 TB/s)"


def profiled_traffic() -> int | None:
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    src_hash = hashlib.sha256(open(DECODE_SOURCE, "rb").read()).hexdigest()[:16]
    m_hash = re.search(r"decode_source_sha256_16:\s*([0-9a-f]+)", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_traffic or m_hash.group(1) != src_hash:
        return None
    return int(m_traffic.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines: list[str] = []
        sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis.split(",")[0].strip().isdigit():
                sel = ["-i", vis.split(",")[0].strip()]
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "20"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_sample(cfg, n_seqs: int):
    """The first n_seqs sequences of the workload (same length draws), on the host."""
    import synth.host as H
    n_seqs = max(cfg.samples, n_seqs // cfg.samples * cfg.samples)
    hw = H.generate(cfg, num_seqs=n_seqs)
    return hw, H.compact_pools(hw)


def time_oracle(cfg, min_seconds: float, n_seqs: int, max_runs: int | None = None) -> dict:
    n_seqs = max(cfg.samples, n_seqs // cfg.samples * cfg.samples)
    """The fp64 oracle, as it stands, on the host cores: one step (new rows
    written, then attention) over a bounded sample of the workload."""
    import oracle
    import synth.host as H
    threads = len(os.sched_getaffinity(0))
    hw, hp0 = cpu_sample(cfg, n_seqs)
    nbytes = workload_bytes(hw.st)["step"]
    times = []
    t_start = time.perf_counter()
    while True:
        hp = H.HostPools(hp0.k_cache.copy(), hp0.v_cache.copy(), hp0.block_tables, hp0.slot_mapping,
                         hp0.copy_pairs, hp0.ids, hp0.seqs, hp0.prefix_tables)
        t0 = time.perf_counter()
        oracle.decode_step(hp, hw, threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= min_seconds or (max_runs and len(times) >= max_runs):
            break
    mean = sum(times) / len(times)
    return {"value": nbytes / mean / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"first {n_seqs} of {cfg.num_seqs} sequences of the same workload "
                       f"({int(hw.st.context_lens.sum())} tokens x {cfg.num_heads} heads), "
                       f"{len(times)} run(s) of one step, {mean * 1e3:.1f} ms each"),
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
    nbytes = workload_bytes(st)
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
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    has_copy, has_new = dw.copy_pairs.numel() > 0, dw.slot_mapping.numel() > 0

    def cache_ops():
        if has_copy:
            pkv.copy_blocks(dw.k_cache, dw.v_cache, dw.copy_pairs, dev_err=err)
        if has_new:
            pkv.reshape_and_cache(dw.new_k, dw.new_v, dw.k_cache, dw.v_cache, dw.slot_mapping, dev_err=err)

    def attention():
        if grouped:
            pkv.paged_attention_decode_grouped(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                               dw.context_lens, cfg.scale, mcl, gs, sb, ws, dev_err=err)
        else:
            pkv.paged_attention_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                       dw.context_lens, cfg.scale, mcl, workspace=ws, dev_err=err)

    def step():
        cache_ops()
        attention()

    launches_per_step = int(has_copy) + int(has_new) + (2 if grouped else 1)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
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
    with ClockSampler(local_rank) as clocks:
        t_wall0 = time.perf_counter()
        for i in range(K):
            flush.fill_(i & 0xFF)        # evict the previous step's lines from L2
            ev[i][0].record(stream)
            cache_ops()
            ev[i][1].record(stream)
            attention()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t_wall0
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    decode_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    cache_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x} in the timed region")

    # end to end through the same API with host buffers: per step, copy the
    # step's inputs from pinned host memory, run the step, read the output back
    dev_in = [t for t in (dw.q, dw.new_k, dw.new_v, dw.slot_mapping, dw.block_tables, dw.context_lens,
                          dw.copy_pairs) if t.numel()]
    if grouped:
        dev_in += [gs, sb]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(10, K // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_total = 0.0
    for i in range(e2e_steps + 3):
        flush.fill_(i & 0xFF)
        if i >= 3:
            e0.record(stream)
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        if i >= 3:
            e1.record(stream)
            e1.synchronize()
            e2e_total += e0.elapsed_time(e1)
    e2e_ms = e2e_total / e2e_steps

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
        cpu = time_oracle(cfg, args.cpu_seconds, args.cpu_seqs)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
    line = {
        "metric": METRIC,
        "value": world * nbytes["step"] / (agg["step_ms"] * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": agg["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic",
        "config": config_json(cfg, st, world, args.attention),
        "seqs_per_s": world * B / (agg["step_ms"] * 1e-3),
        "attention_ms": agg["decode_ms"], "cache_ops_ms": agg["cache_ms"],
        "bytes_per_step": nbytes["step"], "roofline_frac_step": nbytes["step"] / (agg["step_ms"] * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm",
                     "kernel": "pa_group_prologue + pa_decode_grouped_kernel" if grouped else "pa_decode_kernel",
                     "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic() if (cfg.name == WORKLOAD and not grouped) else None,
                     "algorithmic_bytes_per_launch": nbytes["attention"], "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": world * nbytes["step"] / (agg["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": agg["e2e_ms"], "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary(),
        "timed_region_wall_s": wall,
        "kv_memory": kv_memory(cfg),
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
                    help="synthetic workload preset (default: the LLaMA-13B-shaped step)")
    ap.add_argument("--attention", choices=("plain", "grouped"), default="plain",
                    help="grouped: siblings read shared prefix blocks once (copy-on-write workloads)")
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
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
