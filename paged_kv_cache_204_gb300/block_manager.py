"""Python binding of the host block manager (C ABI in include/pkv_block_manager.h).

Argument marshalling only: allocation, reference counting, copy-on-write and
the counters all run in the compiled library ("PagedAttention: the KV cache
was the bottleneck all along", section "Virtual memory for attention").
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import PKV_ERR_OUT_OF_BLOCKS, PkvError, lib

_P, _I32, _I64, _U64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64


class Stats(ctypes.Structure):
    """Counters of pkv_bm_get_stats (see pkv_bm_stats in the header)."""
    _fields_ = [(name, _I64) for name in (
        "num_blocks", "free_blocks", "used_blocks", "shared_blocks", "filled_slots",
        "logical_blocks", "logical_tokens", "live_seqs", "cow_copies")]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


lib.pkv_bm_create.argtypes = [_I32, _I32, _U64, ctypes.POINTER(_P)]
lib.pkv_bm_create.restype = ctypes.c_int
lib.pkv_bm_destroy.argtypes = [_P]
lib.pkv_bm_destroy.restype = None
lib.pkv_bm_add_seq.argtypes = [_P, ctypes.POINTER(_I32)]
lib.pkv_bm_add_seq.restype = ctypes.c_int
lib.pkv_bm_fork.argtypes = [_P, _I32, ctypes.POINTER(_I32)]
lib.pkv_bm_fork.restype = ctypes.c_int
lib.pkv_bm_free_seq.argtypes = [_P, _I32]
lib.pkv_bm_free_seq.restype = ctypes.c_int
lib.pkv_bm_append.argtypes = [_P, _I32, _I32, _P, _P, ctypes.POINTER(_I32)]
lib.pkv_bm_append.restype = ctypes.c_int
lib.pkv_bm_append_batch.argtypes = [_P, _P, _P, _I32, _P, _P, ctypes.POINTER(_I32)]
lib.pkv_bm_append_batch.restype = ctypes.c_int
lib.pkv_bm_beam_step.argtypes = [_P, _P, _P, _I32, _I32, _P, _P, _P, ctypes.POINTER(_I32)]
lib.pkv_bm_beam_step.restype = ctypes.c_int
lib.pkv_bm_beam_step_many.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, ctypes.POINTER(_I32), _P]
lib.pkv_bm_beam_step_many.restype = ctypes.c_int
lib.pkv_bm_seq_info.argtypes = [_P, _I32, ctypes.POINTER(_I64), ctypes.POINTER(_I32)]
lib.pkv_bm_seq_info.restype = ctypes.c_int
lib.pkv_bm_export.argtypes = [_P, _P, _I32, _I32, _P, _P]
lib.pkv_bm_export.restype = ctypes.c_int
lib.pkv_bm_common_prefix.argtypes = [_P, _P, _I32, ctypes.POINTER(_I32)]
lib.pkv_bm_common_prefix.restype = ctypes.c_int
lib.pkv_bm_get_stats.argtypes = [_P, ctypes.POINTER(Stats)]
lib.pkv_bm_get_stats.restype = ctypes.c_int


class OutOfBlocks(PkvError):
    pass


def _check(status: int, what: str) -> None:
    if status == PKV_ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(status, what)
    if status != 0:
        raise PkvError(status, what)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class BlockManager:
    """On-demand block allocator with reference-counted sharing and
    copy-on-write. seed fixes the initial free-block order (0: ascending)."""

    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        h = _P()
        _check(lib.pkv_bm_create(int(num_blocks), int(block_size), int(seed), ctypes.byref(h)), "pkv_bm_create")
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def add_seq(self) -> int:
        out = _I32()
        _check(lib.pkv_bm_add_seq(self._h, ctypes.byref(out)), "pkv_bm_add_seq")
        return out.value

    def fork(self, parent: int) -> int:
        out = _I32()
        _check(lib.pkv_bm_fork(self._h, int(parent), ctypes.byref(out)), "pkv_bm_fork")
        return out.value

    def free_seq(self, seq: int) -> None:
        _check(lib.pkv_bm_free_seq(self._h, int(seq)), "pkv_bm_free_seq")

    def append(self, seq: int, n: int = 1) -> tuple[np.ndarray, tuple[int, int] | None]:
        """Slots (int64 [n]) of the next n tokens of seq, and the
        copy-on-write (src, dst) pair the caller must copy first, if any."""
        slots = np.empty(max(int(n), 0), dtype=np.int64)  # the library rejects n < 0
        pair = np.empty(2, dtype=np.int64)
        ncow = _I32()
        _check(lib.pkv_bm_append(self._h, int(seq), int(n), slots.ctypes.data, pair.ctypes.data,
                                 ctypes.byref(ncow)), "pkv_bm_append")
        return slots, ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def append_batch(self, seqs, counts) -> tuple[np.ndarray, np.ndarray]:
        """Slots (int64, packed in order) for counts[i] more tokens of each
        distinct sequence seqs[i], and the copy-on-write pairs (int64 [k][2])."""
        s, c = _i32(seqs), _i32(counts)
        if s.shape != c.shape:
            raise ValueError("seqs and counts differ in length")
        slots = np.empty(int(c.sum()), dtype=np.int64)
        pairs = np.empty((s.size, 2), dtype=np.int64)
        ncow = _I32()
        _check(lib.pkv_bm_append_batch(self._h, s.ctypes.data, c.ctypes.data, s.size, slots.ctypes.data,
                                       pairs.ctypes.data, ctypes.byref(ncow)), "pkv_bm_append_batch")
        return slots, pairs[:ncow.value].copy()

    def beam_step(self, beams, parents, n_new: int = 1) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """One beam-search step of one request: new beam i continues
        beams[parents[i]] with n_new tokens; beams nobody continues end.
        Returns (new beam sequence ids int32 [W], slots int64 [W * n_new],
        copy-on-write pairs int64 [k][2])."""
        b, p = _i32(beams), _i32(parents)
        if b.shape != p.shape:
            raise ValueError("beams and parents differ in length")
        new = np.empty(b.size, dtype=np.int32)
        slots = np.empty(b.size * max(int(n_new), 0), dtype=np.int64)
        pairs = np.empty((b.size, 2), dtype=np.int64)
        ncow = _I32()
        _check(lib.pkv_bm_beam_step(self._h, b.ctypes.data, p.ctypes.data, b.size, int(n_new), new.ctypes.data,
                                    slots.ctypes.data, pairs.ctypes.data, ctypes.byref(ncow)), "pkv_bm_beam_step")
        return new, slots, pairs[:ncow.value].copy()

    def beam_step_many(self, beams, parents, n_new: int = 1
                       ) -> tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
        """One beam-search step of R requests of W beams at once (beams and
        parents int [R][W]; parents index within their own row). Every
        request's ended beams are released before any request appends.
        Returns (new beam sequence ids int32 [R][W], slots int64
        [R * W * n_new] packed row-major, copy-on-write pairs int64 [k][2],
        blocks shared by all new beams of each request int32 [R])."""
        b, p = _i32(beams), _i32(parents)
        if b.ndim != 2 or b.shape != p.shape:
            raise ValueError("beams and parents must both be [requests][width]")
        R, W = b.shape
        new = np.empty((R, W), dtype=np.int32)
        slots = np.empty(b.size * max(int(n_new), 0), dtype=np.int64)
        pairs = np.empty((b.size, 2), dtype=np.int64)
        shared = np.empty(R, dtype=np.int32)
        ncow = _I32()
        _check(lib.pkv_bm_beam_step_many(self._h, b.ctypes.data, p.ctypes.data, R, W, int(n_new), new.ctypes.data,
                                         slots.ctypes.data, pairs.ctypes.data, ctypes.byref(ncow),
                                         shared.ctypes.data), "pkv_bm_beam_step_many")
        return new, slots, pairs[:ncow.value].copy(), shared

    def seq_info(self, seq: int) -> tuple[int, int]:
        """(length in tokens, table length in blocks) of seq."""
        n, b = _I64(), _I32()
        _check(lib.pkv_bm_seq_info(self._h, int(seq), ctypes.byref(n), ctypes.byref(b)), "pkv_bm_seq_info")
        return n.value, b.value

    def export(self, seqs, max_blocks: int) -> tuple[np.ndarray, np.ndarray]:
        """(block_tables int32 [n][max_blocks] padded with -1, context_lens int32 [n])."""
        s = _i32(seqs)
        bt = np.empty((s.size, int(max_blocks)), dtype=np.int32)
        cl = np.empty(s.size, dtype=np.int32)
        _check(lib.pkv_bm_export(self._h, s.ctypes.data, s.size, int(max_blocks), bt.ctypes.data, cl.ctypes.data),
               "pkv_bm_export")
        return bt, cl

    def common_prefix(self, seqs) -> int:
        """Leading block-table entries the given sequences all share."""
        s = _i32(seqs)
        out = _I32()
        _check(lib.pkv_bm_common_prefix(self._h, s.ctypes.data, s.size, ctypes.byref(out)), "pkv_bm_common_prefix")
        return out.value

    def stats(self) -> dict:
        st = Stats()
        _check(lib.pkv_bm_get_stats(self._h, ctypes.byref(st)), "pkv_bm_get_stats")
        return st.as_dict()


def memory_metrics(stats: dict, block_size: int) -> dict:
    """KV memory figures of a manager state ("PagedAttention: the KV cache was
    the bottleneck all along", section "Virtual memory for attention"):
    waste = allocated slots holding no token / allocated slots (only the
    unfilled tail of each sequence's last block can be empty);
    sharing_saving = 1 - physical blocks in use / blocks the live sequences
    would hold with private copies."""
    alloc = stats["used_blocks"] * block_size
    return {
        "waste_fraction": (alloc - stats["filled_slots"]) / alloc if alloc else 0.0,
        "sharing_saving": 1.0 - stats["used_blocks"] / stats["logical_blocks"] if stats["logical_blocks"] else 0.0,
    }
