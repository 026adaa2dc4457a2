"""fp64 CPU oracle of the PagedAttention decode path.

TEST INFRASTRUCTURE ONLY. The product library never imports, links or calls
this package; only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg (and its ``--impl reference`` arm) do. It shares no code with
the CUDA path: the arithmetic lives in ``pkv_oracle.c`` (plain C99, fp64);
this module only marshals numpy arrays into it.

Semantics follow "PagedAttention: the KV cache was the bottleneck all along",
section "Virtual memory for attention" (fixed-size blocks, a block table from
logical to physical blocks, attention gathering K/V from scattered blocks,
copy-on-write of shared blocks). Each function below states what it computes.

Storage convention shared with the inputs: fp16/bf16 arrays are passed as
their raw 16-bit patterns (``np.uint16``), fp32 as ``np.float32``.

Every function takes an optional ``L``: another build of the same C source
(``load()``), which the tests use to show that the pins catch mistakes planted
in a copy of it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libpkv_oracle.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False, src: str = SOURCE, out: str = _SO) -> str:
    """Compile the oracle C source into a shared library with gcc (plain C99,
    fp64, no FMA contraction so that every host rounds the same way)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
           "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)  # atomic: concurrent builders never see a partial file
    return out


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.orc_paged_attention.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, D, I, I]
    L.orc_paged_attention.restype = I
    L.orc_dense_attention.argtypes = [P, P, P, P, P, I, I, I, I, I, D]
    L.orc_dense_attention.restype = I
    L.orc_paged_attention_chunked.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, D, I]
    L.orc_paged_attention_chunked.restype = I
    L.orc_reshape_and_cache.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    L.orc_reshape_and_cache.restype = I
    L.orc_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I]
    L.orc_copy_blocks.restype = I
    L.orc_decode_f16.argtypes = [ctypes.c_uint16]
    L.orc_decode_f16.restype = D
    L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
    L.orc_decode_bf16.restype = D
    L.orc_decode_f32.argtypes = [ctypes.c_uint32]
    L.orc_decode_f32.restype = D
    L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
    L.orc_decode_e4m3.restype = D
    L.orc_encode_e4m3.argtypes = [D]
    L.orc_encode_e4m3.restype = ctypes.c_uint8
    F = ctypes.c_float
    L.orc_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, F]
    L.orc_reshape_and_cache_fp8.restype = I
    L.orc_paged_attention_fp8.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, D, D, D, I, I]
    L.orc_paged_attention_fp8.restype = I
    L.orc_paged_prefill.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, D, I, I]
    L.orc_paged_prefill.restype = I
    L.orc_encode_f16.argtypes = [D]
    L.orc_encode_f16.restype = ctypes.c_uint16
    L.orc_q4_0_quantize_block.argtypes = [P, P, P]
    L.orc_q4_0_quantize_block.restype = None
    L.orc_q4_0_value.argtypes = [P, I, I]
    L.orc_q4_0_value.restype = D
    L.orc_q4_0_quantize_row.argtypes = [P, I, I, P]
    L.orc_q4_0_quantize_row.restype = I
    L.orc_reshape_and_cache_q4_0.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    L.orc_reshape_and_cache_q4_0.restype = I
    L.orc_paged_attention_q4_0.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, D, I, I]
    L.orc_paged_attention_q4_0.restype = I
    return L


_default = None


def lib() -> ctypes.CDLL:
    global _default
    if _default is None:
        _default = _bind(ctypes.CDLL(build()))
    return _default


def load(so_path: str) -> ctypes.CDLL:
    """Load another build of the oracle source."""
    return _bind(ctypes.CDLL(so_path))


def _ptr(a: np.ndarray) -> int:
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle inputs must be C-contiguous")
    return a.ctypes.data


def _check_store(a: np.ndarray, dtype: str, name: str) -> None:
    want = np.float32 if dtype == "f32" else np.uint16
    if a.dtype != want:
        raise TypeError(f"{name}: {dtype} storage must be {np.dtype(want).name}, got {a.dtype}")


def decode_elements(bits: np.ndarray, dtype: str, L=None) -> np.ndarray:
    """Decode stored elements to float64 with the oracle's own decoders."""
    L = L or lib()
    f = {"f16": L.orc_decode_f16, "bf16": L.orc_decode_bf16, "f32": L.orc_decode_f32}[dtype]
    flat = np.ascontiguousarray(bits).reshape(-1)
    if dtype == "f32":
        flat = flat.view(np.uint32)
    return np.array([f(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, *, scale, num_heads,
                    num_kv_heads, head_dim, block_size, dtype, threads: int = 1,
                    seqs: tuple[int, int] | None = None, L=None) -> np.ndarray:
    """Decode attention over a paged cache, fp64: out[s][h][:] =
    softmax_t(scale * q[s][h] . K_t) . V_t over the first context_lens[s] tokens,
    token t read from block block_tables[s][t // block_size], row t % block_size,
    kv head h // (num_heads // num_kv_heads).

    ``threads`` > 1 splits the sequence range over threads (ctypes releases the
    GIL during the C call); the arithmetic per (s, h) is unchanged.
    Returns float64 [num_seqs, num_heads, head_dim] (rows outside ``seqs`` are 0).
    """
    L = L or lib()
    for a, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_store(a, dtype, n)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = cl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    num_blocks = k_cache.shape[0]
    out = np.zeros((B, num_heads, head_dim), dtype=np.float64)
    lo, hi = seqs if seqs is not None else (0, B)

    def run(a, b):
        rc = L.orc_paged_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                   bt.shape[1], _ptr(cl), B, num_heads, num_kv_heads, head_dim,
                                   block_size, num_blocks, DTYPE_CODE[dtype], float(scale), a, b)
        if rc != 0:
            raise ValueError(f"orc_paged_attention failed with code {rc}")

    if threads <= 1 or hi - lo <= 1:
        run(lo, hi)
    else:
        # contiguous runs of sequences with about the same number of tokens each
        lens = np.maximum(cl[lo:hi].astype(np.int64), 1)
        cuts = np.searchsorted(np.cumsum(lens), np.linspace(0, lens.sum(), threads + 1)[1:-1])
        bounds = sorted(set([lo] + [min(hi, lo + int(c) + 1) for c in cuts] + [hi]))
        pieces = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        with ThreadPoolExecutor(max_workers=len(pieces)) as ex:
            list(ex.map(lambda ab: run(*ab), pieces))
    return out


def paged_attention_chunked(q, k_cache, v_cache, block_tables, context_lens, *, scale,
                            num_heads, num_kv_heads, head_dim, block_size, dtype,
                            chunk: int, L=None) -> np.ndarray:
    """The same attention evaluated chunk by chunk (each chunk keeps its own
    max, exp-sum and normalised output) and combined with the log-sum-exp rule."""
    L = L or lib()
    for a, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_store(a, dtype, n)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = cl.shape[0]
    out = np.zeros((B, num_heads, head_dim), dtype=np.float64)
    rc = L.orc_paged_attention_chunked(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1], _ptr(cl), B,
        num_heads, num_kv_heads, head_dim, block_size, k_cache.shape[0], DTYPE_CODE[dtype],
        float(scale), int(chunk))
    if rc != 0:
        raise ValueError(f"orc_paged_attention_chunked failed with code {rc}")
    return out


def dense_attention(q, k, v, seq_start, *, scale, num_heads, num_kv_heads, head_dim,
                    dtype, L=None) -> np.ndarray:
    """Attention over K/V laid out contiguously: k, v are
    [total_tokens, num_kv_heads, head_dim]; sequence s owns rows
    seq_start[s]:seq_start[s+1]. No block table involved."""
    L = L or lib()
    for a, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_store(a, dtype, n)
    st = np.ascontiguousarray(seq_start, dtype=np.int64)
    B = st.shape[0] - 1
    out = np.zeros((B, num_heads, head_dim), dtype=np.float64)
    rc = L.orc_dense_attention(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(st), B, num_heads,
                               num_kv_heads, head_dim, DTYPE_CODE[dtype], float(scale))
    if rc != 0:
        raise ValueError(f"orc_dense_attention failed with code {rc}")
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, *, num_kv_heads, head_dim,
                      block_size, dtype, L=None) -> int:
    """In place on k_cache/v_cache: token t's rows go to slot slot_mapping[t]
    (block slot // block_size, row slot % block_size); negative slots are
    skipped. Returns the number of out-of-range slots (not written)."""
    L = L or lib()
    for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_store(a, dtype, n)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = L.orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                 sm.shape[0], num_kv_heads, head_dim, block_size,
                                 k_cache.shape[0], DTYPE_CODE[dtype])
    if rc < 0:
        raise ValueError(f"orc_reshape_and_cache failed with code {rc}")
    return rc


def copy_blocks(k_cache, v_cache, block_pairs, *, num_kv_heads, head_dim, block_size,
                dtype, L=None) -> int:
    """In place: for each (src, dst) pair, block dst of both pools becomes a
    copy of block src. Returns the number of pairs skipped as out of range."""
    L = L or lib()
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_store(a, dtype, n)
    pairs = np.ascontiguousarray(block_pairs, dtype=np.int64).reshape(-1, 2)
    rc = L.orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0],
                           num_kv_heads, head_dim, block_size, k_cache.shape[0],
                           DTYPE_CODE[dtype])
    if rc < 0:
        raise ValueError(f"orc_copy_blocks failed with code {rc}")
    return rc


def decode_step(hp, hw, threads: int = 1, L=None) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One decode step on host pools `hp` (synth.host.HostPools) of workload
    `hw`, in the step's order: copy-on-write copies, then the new K/V rows,
    then attention, for the sequences hp serves (out row i = sequence
    hp.seqs[i]). Mutates hp's pools; returns (out, k_cache, v_cache)."""
    cfg = hw.cfg
    kw = dict(num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim, block_size=cfg.block_size,
              dtype=cfg.dtype, L=L)
    if hp.copy_pairs.size:
        copy_blocks(hp.k_cache, hp.v_cache, hp.copy_pairs, **kw)
    if hp.slot_mapping.size:
        reshape_and_cache(hw.new_k, hw.new_v, hp.k_cache, hp.v_cache, hp.slot_mapping, **kw)
    q = np.ascontiguousarray(hw.q[hp.seqs])
    out = paged_attention(q, hp.k_cache, hp.v_cache, hp.block_tables, hw.st.context_lens[hp.seqs],
                          scale=cfg.scale, num_heads=cfg.num_heads, num_kv_heads=cfg.num_kv_heads,
                          head_dim=cfg.head_dim, block_size=cfg.block_size, dtype=cfg.dtype,
                          threads=threads, L=L)
    return out, hp.k_cache, hp.v_cache


# ---- fp8 (e4m3) KV cache ------------------------------------------------------

def decode_e4m3(codes: np.ndarray, L=None) -> np.ndarray:
    """E4M3 codes (uint8) -> float64, with the oracle's own decoder."""
    L = L or lib()
    flat = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([L.orc_decode_e4m3(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))


def encode_e4m3(values: np.ndarray, L=None) -> np.ndarray:
    """float64 values -> nearest E4M3 codes (ties to even, saturating)."""
    L = L or lib()
    flat = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    return np.array([L.orc_encode_e4m3(float(x)) for x in flat], dtype=np.uint8).reshape(np.shape(values))


def reshape_and_cache_fp8(k, v, k_cache, v_cache, slot_mapping, *, num_kv_heads, head_dim, block_size,
                          src_dtype, k_scale, v_scale, L=None) -> int:
    """In place on the uint8 pools: token t's rows, divided by the scale in
    binary32 and rounded to E4M3, go to slot slot_mapping[t]. Returns the
    number of out-of-range slots."""
    L = L or lib()
    for a, n in ((k, "k"), (v, "v")):
        _check_store(a, src_dtype, n)
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        if a.dtype != np.uint8:
            raise TypeError(f"{n}: e4m3 pools must be uint8, got {a.dtype}")
    sl = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = L.orc_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sl), sl.shape[0],
                                     num_kv_heads, head_dim, block_size, k_cache.shape[0], DTYPE_CODE[src_dtype],
                                     float(k_scale), float(v_scale))
    if rc < 0:
        raise ValueError(f"orc_reshape_and_cache_fp8 failed with code {rc}")
    return rc


def paged_attention_fp8(q, k_cache, v_cache, block_tables, context_lens, *, scale, k_scale, v_scale, num_heads,
                        num_kv_heads, head_dim, block_size, q_dtype, threads: int = 1, L=None) -> np.ndarray:
    """Decode attention over E4M3 pools, fp64: paged_attention with K
    elements k_scale * code and V elements v_scale * code."""
    L = L or lib()
    _check_store(q, q_dtype, "q")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = cl.shape[0]
    out = np.zeros((B, num_heads, head_dim), dtype=np.float64)

    def run(lo, hi):
        return L.orc_paged_attention_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                                         _ptr(cl), B, num_heads, num_kv_heads, head_dim, block_size,
                                         k_cache.shape[0], DTYPE_CODE[q_dtype], float(scale), float(k_scale),
                                         float(v_scale), lo, hi)

    n = max(1, min(threads, B))
    cuts = [B * i // n for i in range(n + 1)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        rcs = list(ex.map(lambda i: run(cuts[i], cuts[i + 1]), range(n)))
    if any(rc != 0 for rc in rcs):
        raise ValueError(f"orc_paged_attention_fp8 failed with codes {rcs}")
    return out


# ---- 4-bit (q4_0) KV cache -----------------------------------------------------

def q4_0_row_bytes(head_dim: int) -> int:
    """Bytes of one cache row of head_dim values: head_dim / 32 binary16
    scales, then head_dim / 2 code bytes."""
    return head_dim // 16 * 9


def encode_f16(values: np.ndarray, L=None) -> np.ndarray:
    """float64 values -> nearest binary16 bit patterns (ties to even)."""
    L = L or lib()
    flat = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    return np.array([L.orc_encode_f16(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(values))


def q4_0_quantize_block(x: np.ndarray, L=None):
    """32 binary32 values -> (scale bits as uint16, 16 code bytes)."""
    L = L or lib()
    xb = np.ascontiguousarray(x, dtype=np.float32)
    if xb.shape != (32,):
        raise ValueError("a q4_0 block holds 32 values")
    d = np.zeros(1, dtype=np.uint16)
    qs = np.zeros(16, dtype=np.uint8)
    L.orc_q4_0_quantize_block(_ptr(xb), _ptr(d), _ptr(qs))
    return int(d[0]), qs


def q4_0_quantize_row(src: np.ndarray, src_dtype: str, L=None) -> np.ndarray:
    """One row of head_dim binary16 / bfloat16 values (uint16 bits) -> its
    9 head_dim / 16 cache bytes."""
    L = L or lib()
    _check_store(src, src_dtype, "src")
    sb = np.ascontiguousarray(src).reshape(-1)
    row = np.zeros(q4_0_row_bytes(sb.shape[0]), dtype=np.uint8)
    rc = L.orc_q4_0_quantize_row(_ptr(sb), DTYPE_CODE[src_dtype], sb.shape[0], _ptr(row))
    if rc != 0:
        raise ValueError(f"orc_q4_0_quantize_row failed with code {rc}")
    return row


def q4_0_values(row: np.ndarray, head_dim: int, L=None) -> np.ndarray:
    """The head_dim values a q4_0 cache row reads back as (float64)."""
    L = L or lib()
    rb = np.ascontiguousarray(row, dtype=np.uint8).reshape(-1)
    return np.array([L.orc_q4_0_value(_ptr(rb), head_dim, d) for d in range(head_dim)], dtype=np.float64)


def reshape_and_cache_q4_0(k, v, k_cache, v_cache, slot_mapping, *, num_kv_heads, head_dim, block_size,
                           src_dtype, L=None) -> int:
    """In place on the uint8 pools [num_blocks][kv_heads][block_size][9 D / 16]:
    token t's rows, quantised to q4_0 blocks, go to slot slot_mapping[t].
    Returns the number of out-of-range slots."""
    L = L or lib()
    for a, n in ((k, "k"), (v, "v")):
        _check_store(a, src_dtype, n)
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        if a.dtype != np.uint8:
            raise TypeError(f"{n}: q4_0 pools must be uint8, got {a.dtype}")
    sl = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = L.orc_reshape_and_cache_q4_0(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sl), sl.shape[0],
                                      num_kv_heads, head_dim, block_size, k_cache.shape[0], DTYPE_CODE[src_dtype])
    if rc < 0:
        raise ValueError(f"orc_reshape_and_cache_q4_0 failed with code {rc}")
    return rc


def paged_attention_q4_0(q, k_cache, v_cache, block_tables, context_lens, *, scale, num_heads, num_kv_heads,
                         head_dim, block_size, q_dtype, threads: int = 1, L=None) -> np.ndarray:
    """Decode attention over q4_0 pools, fp64: paged_attention with every
    K and V element read back as d * (q - 8)."""
    L = L or lib()
    _check_store(q, q_dtype, "q")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = cl.shape[0]
    out = np.zeros((B, num_heads, head_dim), dtype=np.float64)

    def run(lo, hi):
        return L.orc_paged_attention_q4_0(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                          bt.shape[1], _ptr(cl), B, num_heads, num_kv_heads, head_dim,
                                          block_size, k_cache.shape[0], DTYPE_CODE[q_dtype], float(scale), lo, hi)

    n = max(1, min(threads, B))
    cuts = [B * i // n for i in range(n + 1)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        rcs = list(ex.map(lambda i: run(cuts[i], cuts[i + 1]), range(n)))
    if any(rc != 0 for rc in rcs):
        raise ValueError(f"orc_paged_attention_q4_0 failed with codes {rcs}")
    return out


# ---- paged prefill -------------------------------------------------------------

def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, *, scale, num_heads,
                  num_kv_heads, head_dim, block_size, dtype, threads: int = 1, L=None) -> np.ndarray:
    """Causal attention of each sequence's last n = query_start[s+1] -
    query_start[s] tokens over its paged context (query i at position
    context_lens[s] - n + i sees tokens 0 .. that position). q is packed
    [total_queries, num_heads, head_dim]; returns float64 of the same shape."""
    L = L or lib()
    for a, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_store(a, dtype, n)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    B = cl.shape[0]
    out = np.zeros((q.shape[0], num_heads, head_dim), dtype=np.float64)

    def run(lo, hi):
        return L.orc_paged_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1], _ptr(cl),
                                   _ptr(qs), B, num_heads, num_kv_heads, head_dim, block_size, k_cache.shape[0],
                                   DTYPE_CODE[dtype], float(scale), lo, hi)

    n = max(1, min(threads, B))
    cuts = [B * i // n for i in range(n + 1)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        rcs = list(ex.map(lambda i: run(cuts[i], cuts[i + 1]), range(n)))
    if any(rc != 0 for rc in rcs):
        raise ValueError(f"orc_paged_prefill failed with codes {rcs}")
    return out
