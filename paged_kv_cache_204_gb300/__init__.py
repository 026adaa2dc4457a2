"""Python binding of the paged KV-cache library (C ABI in include/pkv.h).

Argument marshalling only: every entry point forwards device pointers, sizes
and the current CUDA stream to the compiled library, which does all the work
in its own kernels. There is no fallback: importing this package without the
built library (``python -m paged_kv_cache_204_gb300.build`` or
``__graft_entry__.build()``) raises ImportError.

Functions mirror the C entry points:
  reshape_and_cache       -> pkv_reshape_and_cache
  copy_blocks             -> pkv_copy_blocks
  paged_attention_decode  -> pkv_paged_attention_decode
  decode_workspace_bytes  -> pkv_decode_workspace_bytes
  paged_attention_decode_grouped  -> pkv_paged_attention_decode_grouped
  reshape_and_cache_fp8, paged_attention_decode_fp8  -> the fp8 (e4m3) cache entry points
  reshape_and_cache_q4_0, paged_attention_decode_q4_0, copy_blocks_q4_0
                          -> the 4-bit (q4_0) cache entry points
  paged_attention_prefill -> pkv_paged_attention_prefill
  decode_grouped_workspace_bytes  -> pkv_decode_grouped_workspace_bytes
  set_wait_timeout_ns / get_wait_timeout_ns, status_string, version
The host block manager (include/pkv_block_manager.h) is wrapped by
``paged_kv_cache_204_gb300.block_manager.BlockManager``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LIB_PATH = _build.LIB

if not os.path.exists(LIB_PATH):
    raise ImportError(f"paged_kv_cache_204_gb300: compiled library missing at {LIB_PATH}; "
                      "build it with `python -m paged_kv_cache_204_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA, PKV_ERR_OUT_OF_BLOCKS = range(6)
DEV_ERR_BLOCK_ID, DEV_ERR_SLOT, DEV_ERR_CONTEXT_LEN, DEV_ERR_TIMEOUT, DEV_ERR_PAIR = 1, 2, 4, 8, 16
DEV_ERR_GROUP = 32
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.uint8: 3}  # uint8: e4m3 codes
PKV_FP8_E4M3 = 3
PKV_Q4_0 = 4

_P, _I, _I64, _U64, _F, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                               ctypes.c_float, ctypes.c_size_t)
lib.pkv_status_string.argtypes = [_I]
lib.pkv_status_string.restype = ctypes.c_char_p
lib.pkv_version.argtypes = []
lib.pkv_version.restype = _I
lib.pkv_set_wait_timeout_ns.argtypes = [_U64]
lib.pkv_set_wait_timeout_ns.restype = None
lib.pkv_get_wait_timeout_ns.argtypes = []
lib.pkv_get_wait_timeout_ns.restype = _U64
lib.pkv_decode_workspace_bytes.argtypes = [_I, _I, _I, _I]
lib.pkv_decode_workspace_bytes.restype = _SZ
lib.pkv_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]
lib.pkv_reshape_and_cache.restype = _I
lib.pkv_copy_blocks.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]
lib.pkv_copy_blocks.restype = _I
lib.pkv_paged_attention_decode.argtypes = [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I,
                                           _I, _I, _P, _SZ, _P, _P]
lib.pkv_paged_attention_decode.restype = _I
lib.pkv_paged_attention_decode_grouped.argtypes = [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I,
                                                   _I, _I, _P, _P, _I, _I, _P, _SZ, _P, _P]
lib.pkv_paged_attention_decode_grouped.restype = _I
lib.pkv_decode_grouped_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
lib.pkv_decode_grouped_workspace_bytes.restype = _SZ
lib.pkv_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _P, _P]
lib.pkv_reshape_and_cache_fp8.restype = _I
lib.pkv_paged_attention_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _F, _F, _F, _I, _I, _I, _I, _I, _I, _I,
                                               _I, _I, _P, _SZ, _P, _P]
lib.pkv_paged_attention_decode_fp8.restype = _I
lib.pkv_reshape_and_cache_q4_0.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]
lib.pkv_reshape_and_cache_q4_0.restype = _I
lib.pkv_paged_attention_decode_q4_0.argtypes = [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                                _P, _SZ, _P, _P]
lib.pkv_paged_attention_decode_q4_0.restype = _I
lib.pkv_paged_attention_prefill.argtypes = [_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                              _P, _P]
lib.pkv_paged_attention_prefill.restype = _I
lib.pkv_paged_attention_decode_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I,
                                                   _I, _I, _I, _P, _P]
lib.pkv_paged_attention_decode_noalloc.restype = _I
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # PKV_NOALLOC_SCRATCH_BYTES


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


def status_string(status: int) -> str:
    return lib.pkv_status_string(int(status)).decode()


def version() -> int:
    return lib.pkv_version()


def set_wait_timeout_ns(ns: int) -> None:
    lib.pkv_set_wait_timeout_ns(int(ns))


def get_wait_timeout_ns() -> int:
    return lib.pkv_get_wait_timeout_ns()


def decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int) -> int:
    return lib.pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, dev_err: torch.Tensor | None = None,
                      stream=None) -> None:
    """k, v [T, Hkv, D]; k_cache, v_cache [num_blocks, Hkv, block_size, D];
    slot_mapping int64 [T] (all on the GPU)."""
    T, Hkv, D = k.shape
    nb, _, bs, _ = k_cache.shape
    _check(lib.pkv_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                     T, Hkv, D, bs, nb, DTYPE_CODE[k_cache.dtype], _ptr(dev_err),
                                     _stream(stream)), "pkv_reshape_and_cache")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_pairs: torch.Tensor,
                dev_err: torch.Tensor | None = None, stream=None) -> None:
    """block_pairs int64 [n, 2] (src, dst) on the GPU."""
    nb, Hkv, bs, D = k_cache.shape
    n = block_pairs.numel() // 2
    _check(lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), n, Hkv, D, bs, nb,
                               DTYPE_CODE[k_cache.dtype], _ptr(dev_err), _stream(stream)),
           "pkv_copy_blocks")


def paged_attention_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, max_context_len: int,
                           workspace: torch.Tensor | None = None,
                           dev_err: torch.Tensor | None = None, stream=None) -> None:
    """out, q [B, H, D]; caches [num_blocks, Hkv, block_size, D]; block_tables
    int32 [B, max_blocks_per_seq]; context_lens int32 [B]; workspace: a
    zero-initialised device buffer of decode_workspace_bytes() bytes (reused
    across calls; the library leaves its counters zero)."""
    B, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), H, Hkv, D, bs, B, block_tables.shape[1], nb, int(max_context_len),
        DTYPE_CODE[q.dtype], _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)),
        "pkv_paged_attention_decode")


def paged_attention_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float, max_context_len: int,
                                   dev_err: torch.Tensor | None = None, stream=None) -> None:
    """paged_attention_decode without a workspace: for callers that cannot
    allocate device memory, the library keeps the partial results of long
    contexts in its own fixed 32 MiB device array (sizes that need more are
    rejected). Calls that overlap on the GPU share that array and race."""
    B, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    _check(lib.pkv_paged_attention_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), H, Hkv, D, bs, B, block_tables.shape[1], nb, int(max_context_len),
        DTYPE_CODE[q.dtype], _ptr(dev_err), _stream(stream)),
        "pkv_paged_attention_decode_noalloc")


def reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                          dev_err: torch.Tensor | None = None, stream=None) -> None:
    """k, v [T, Hkv, D] fp16/bf16; k_cache, v_cache uint8 [num_blocks, Hkv,
    block_size, D] of e4m3 codes; element x is stored as e4m3(x / scale)."""
    T, Hkv, D = k.shape
    nb, _, bs, _ = k_cache.shape
    _check(lib.pkv_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, Hkv,
                                         D, bs, nb, DTYPE_CODE[k.dtype], float(k_scale), float(v_scale), _ptr(dev_err),
                                         _stream(stream)), "pkv_reshape_and_cache_fp8")


def paged_attention_decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                               k_scale: float, v_scale: float, max_context_len: int,
                               workspace: torch.Tensor | None = None, dev_err: torch.Tensor | None = None,
                               stream=None) -> None:
    """paged_attention_decode over uint8 pools of e4m3 codes: K values are
    k_scale * code, V values v_scale * code; q, out fp16/bf16."""
    B, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), float(k_scale), float(v_scale), H, Hkv, D, bs, B, block_tables.shape[1], nb,
        int(max_context_len), DTYPE_CODE[q.dtype], _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)),
        "pkv_paged_attention_decode_fp8")


def q4_0_row_bytes(head_dim: int) -> int:
    """Bytes of one q4_0 cache row: head_dim / 32 binary16 scales, then
    head_dim / 2 code bytes."""
    return head_dim // 16 * 9


def reshape_and_cache_q4_0(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           slot_mapping: torch.Tensor, dev_err: torch.Tensor | None = None, stream=None) -> None:
    """k, v [T, Hkv, D] fp16/bf16; k_cache, v_cache uint8 [num_blocks, Hkv,
    block_size, 9 D / 16] of q4_0 rows."""
    T, Hkv, D = k.shape
    nb, _, bs, _ = k_cache.shape
    _check(lib.pkv_reshape_and_cache_q4_0(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T,
                                          Hkv, D, bs, nb, DTYPE_CODE[k.dtype], _ptr(dev_err), _stream(stream)),
           "pkv_reshape_and_cache_q4_0")


def paged_attention_decode_q4_0(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                max_context_len: int, workspace: torch.Tensor | None = None,
                                dev_err: torch.Tensor | None = None, stream=None) -> None:
    """paged_attention_decode over uint8 pools of q4_0 rows; q, out fp16/bf16."""
    B, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_q4_0(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), H, Hkv, D, bs, B, block_tables.shape[1], nb, int(max_context_len), DTYPE_CODE[q.dtype],
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)), "pkv_paged_attention_decode_q4_0")


def copy_blocks_q4_0(k_cache: torch.Tensor, v_cache: torch.Tensor, block_pairs: torch.Tensor, head_dim: int,
                     dev_err: torch.Tensor | None = None, stream=None) -> None:
    """copy_blocks over uint8 pools of q4_0 rows of head_dim values."""
    nb, Hkv, bs, _ = k_cache.shape
    n = block_pairs.numel() // 2
    _check(lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), n, Hkv, int(head_dim), bs, nb,
                               PKV_Q4_0, _ptr(dev_err), _stream(stream)), "pkv_copy_blocks")


def paged_attention_prefill(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, query_start: torch.Tensor,
                            scale: float, max_query_len: int, dev_err: torch.Tensor | None = None,
                            stream=None) -> None:
    """Causal attention of each sequence's last n = query_start[s+1] -
    query_start[s] tokens over its paged context. q, out [total_queries, H, D]
    (fp16/bf16) packed by sequence; query_start int32 [B+1] (on the GPU)."""
    _, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    B = context_lens.numel()
    _check(lib.pkv_paged_attention_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), _ptr(query_start),
        float(scale), H, Hkv, D, bs, B, block_tables.shape[1], nb, int(max_query_len), DTYPE_CODE[q.dtype],
        _ptr(dev_err), _stream(stream)), "pkv_paged_attention_prefill")


def decode_grouped_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                                   num_groups: int) -> int:
    return lib.pkv_decode_grouped_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, num_groups)


def paged_attention_decode_grouped(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float, max_context_len: int,
                                   group_start: torch.Tensor, shared_blocks: torch.Tensor,
                                   workspace: torch.Tensor, dev_err: torch.Tensor | None = None,
                                   stream=None) -> None:
    """paged_attention_decode for groups of sequences sharing prefix blocks:
    group g = sequences group_start[g]:group_start[g+1] (int32 [G+1]) whose
    first shared_blocks[g] (int32 [G]) block-table entries are the same
    physical blocks. workspace: zero-initialised, decode_grouped_workspace_bytes()."""
    B, H, D = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    G = shared_blocks.numel()
    _check(lib.pkv_paged_attention_decode_grouped(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), H, Hkv, D, bs, B, block_tables.shape[1], nb, int(max_context_len),
        _ptr(group_start), _ptr(shared_blocks), G, DTYPE_CODE[q.dtype], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)),
        "pkv_paged_attention_decode_grouped")


def new_grouped_workspace(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                          num_groups: int, device="cuda") -> torch.Tensor:
    n = decode_grouped_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, num_groups)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def new_workspace(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                  device="cuda") -> torch.Tensor | None:
    """A zeroed workspace of the size the decode call needs (None if 0)."""
    n = decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None
