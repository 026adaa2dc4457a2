"""The C-ABI library (no GPU needed): it loads, exports exactly the entry
points include/*.h declares, and its host-side checks reject bad arguments
before anything would reach the device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_204_gb300 as m
    return m


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_match_header(pkv):
    declared = _declared()
    assert {"pkv_paged_attention_decode", "pkv_reshape_and_cache", "pkv_copy_blocks"} <= declared
    for name in declared:
        assert hasattr(pkv.lib, name), f"{name} declared but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_[a-z0-9_]+)$", out, flags=re.M))
    assert exported == declared, f"exported {exported ^ declared} differ from the header"


def test_status_strings_and_version(pkv):
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(3) == "PKV_ERR_WORKSPACE"
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"
    assert pkv.version() >= 100


def test_timeout_setting_round_trip(pkv):
    old = pkv.get_wait_timeout_ns()
    assert old == 10 ** 9
    pkv.set_wait_timeout_ns(12345)
    assert pkv.get_wait_timeout_ns() == 12345
    pkv.set_wait_timeout_ns(old)


def test_workspace_size(pkv):
    slots = 4096 * 2 * 4
    align = lambda x: -(-x // 256) * 256
    for B, H, D in ((128, 40, 128), (8, 32, 128), (4, 2, 64)):
        expect = align(B * H * 4) + align(slots * 8) + slots * D * 4
        assert pkv.decode_workspace_bytes(B, H, D, 2048) == expect
        assert pkv.decode_workspace_bytes(B, H, D, 1) == expect     # independent of context length
    assert pkv.decode_workspace_bytes(0, 40, 128, 2048) == 0
    assert pkv.decode_workspace_bytes(128, 40, 128, 2048) <= pkv.NOALLOC_SCRATCH_BYTES


FAKE = 0x10000  # aligned, never dereferenced: every call below returns before any device work


def _decode(pkv, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, scale=0.1, H=8, Hkv=8, D=128, bs=16,
             B=4, MB=8, NB=100, mcl=128, dtype=1, ws=None, ws_bytes=0, err=None, stream=None)
    a.update(kw)
    return pkv.lib.pkv_paged_attention_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["scale"],
                                              a["H"], a["Hkv"], a["D"], a["bs"], a["B"], a["MB"], a["NB"],
                                              a["mcl"], a["dtype"], a["ws"], a["ws_bytes"], a["err"],
                                              a["stream"])


def test_decode_host_checks(pkv):
    INV, UNS, WS, OK = pkv.PKV_ERR_INVALID_ARG, pkv.PKV_ERR_UNSUPPORTED, pkv.PKV_ERR_WORKSPACE, pkv.PKV_OK
    assert _decode(pkv, B=0) == OK                       # nothing to do
    assert _decode(pkv, q=None) == INV
    assert _decode(pkv, out=FAKE + 8) == INV             # misaligned
    assert _decode(pkv, Hkv=3) == INV                    # 8 % 3 != 0
    assert _decode(pkv, mcl=129) == INV                  # > MB * bs
    assert _decode(pkv, B=-1) == INV
    assert _decode(pkv, scale=float("nan")) == INV
    assert _decode(pkv, D=96) == UNS
    assert _decode(pkv, bs=64) == UNS
    assert _decode(pkv, dtype=7) == UNS
    assert _decode(pkv, B=70000, MB=1, mcl=16) == UNS
    big = dict(MB=200, mcl=3000)
    assert _decode(pkv, **big) == WS                     # a workspace is always needed
    need = pkv.decode_workspace_bytes(4, 8, 128, 3000)
    assert _decode(pkv, ws=FAKE, ws_bytes=need - 1, **big) == WS
    assert _decode(pkv, ws=FAKE + 4, ws_bytes=need, **big) == INV


def test_cache_op_host_checks(pkv):
    L = pkv.lib
    INV, UNS, OK = pkv.PKV_ERR_INVALID_ARG, pkv.PKV_ERR_UNSUPPORTED, pkv.PKV_OK
    # (k, v, k_cache, v_cache, slots, T, Hkv, D, bs, NB, dtype, err, stream)
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 128, 16, 10, 2, None, None) == OK
    assert L.pkv_reshape_and_cache(None, FAKE, FAKE, FAKE, FAKE, 3, 4, 128, 16, 10, 2, None, None) == INV
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 3, 4, 128, 16, 10, 2, None, None) == INV
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 80, 16, 10, 2, None, None) == UNS
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 128, 16, 10, 2, None, None) == INV
    # (k_cache, v_cache, pairs, n, Hkv, D, bs, NB, dtype, err, stream)
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 128, 16, 10, 1, None, None) == OK
    assert L.pkv_copy_blocks(FAKE, None, FAKE, 2, 4, 128, 16, 10, 1, None, None) == INV
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 2, 4, 128, 12, 10, 1, None, None) == UNS
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 2, 0, 128, 16, 10, 1, None, None) == INV


def test_fp8_host_checks(pkv):
    L = pkv.lib
    INV, UNS, OK = pkv.PKV_ERR_INVALID_ARG, pkv.PKV_ERR_UNSUPPORTED, pkv.PKV_OK
    # (k, v, k_cache, v_cache, slots, T, Hkv, D, bs, NB, src_dtype, k_scale, v_scale, err, stream)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 128, 16, 10, 1, 0.5, 0.5, None, None]

    def rc(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.pkv_reshape_and_cache_fp8(*a)
    assert rc(a5=0) == OK
    assert rc(a11=0.0) == INV and rc(a12=float("inf")) == INV and rc(a11=-1.0) == INV
    assert rc(a10=0) == UNS            # binary32 rows: not taken
    assert rc(a10=3) == UNS            # e4m3 rows: not a source type
    assert rc(a0=None) == INV and rc(a4=FAKE + 4) == INV
    # decode: (out, q, k, v, bt, cl, scale, k_scale, v_scale, H, Hkv, D, bs, B, MB, NB, mcl, dtype, ws, ws_bytes, err, s)
    d = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 0.5, 0.5, 8, 8, 128, 16, 4, 8, 100, 128, 1, None, 0, None, None]

    def dc(**kw):
        a = list(d)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.pkv_paged_attention_decode_fp8(*a)
    assert dc(a13=0) == OK
    assert dc(a7=0.0) == INV and dc(a8=float("nan")) == INV
    assert dc(a17=0) == UNS            # binary32 queries: not taken
    assert dc(a17=3) == UNS            # e4m3 queries: not taken
    assert dc() == pkv.PKV_ERR_WORKSPACE
    # block copies take the 1-byte element
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 128, 16, 10, 3, None, None) == OK
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 2, 4, 128, 16, 10, 5, None, None) == UNS


def test_q4_0_host_checks(pkv):
    L = pkv.lib
    INV, UNS, OK = pkv.PKV_ERR_INVALID_ARG, pkv.PKV_ERR_UNSUPPORTED, pkv.PKV_OK
    # (k, v, k_cache, v_cache, slots, T, Hkv, D, bs, NB, src_dtype, err, stream)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 128, 16, 10, 1, None, None]

    def rc(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.pkv_reshape_and_cache_q4_0(*a)
    assert rc(a5=0) == OK
    assert rc(a10=0) == UNS and rc(a10=3) == UNS and rc(a10=4) == UNS  # only 16-bit sources
    assert rc(a7=96) == UNS and rc(a8=4) == UNS
    assert rc(a0=None) == INV and rc(a2=FAKE + 8) == INV and rc(a4=FAKE + 4) == INV and rc(a6=0) == INV
    # decode: (out, q, k, v, bt, cl, scale, H, Hkv, D, bs, B, MB, NB, mcl, dtype, ws, ws_bytes, err, s)
    d = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 8, 2, 128, 16, 4, 8, 100, 128, 2, None, 0, None, None]

    def dc(**kw):
        a = list(d)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.pkv_paged_attention_decode_q4_0(*a)
    assert dc(a11=0) == OK
    assert dc(a15=0) == UNS            # binary32 queries: not taken
    assert dc(a9=80) == UNS            # head_dim outside {64, 128}
    assert dc(a7=5) == INV             # query heads not a multiple of kv heads
    assert dc(a6=float("inf")) == INV
    assert dc() == pkv.PKV_ERR_WORKSPACE
    assert dc(a16=FAKE + 8, a17=1 << 30) == INV  # misaligned workspace
    # block copies: q4_0 rows of 9 D / 16 bytes
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 128, 16, 10, 4, None, None) == OK
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 48, 16, 10, 4, None, None) == UNS
    assert pkv.q4_0_row_bytes(128) == 72 and pkv.q4_0_row_bytes(64) == 36


def test_prefill_host_checks(pkv):
    L = pkv.lib
    INV, UNS, OK = pkv.PKV_ERR_INVALID_ARG, pkv.PKV_ERR_UNSUPPORTED, pkv.PKV_OK
    # (out, q, k, v, bt, cl, query_start, scale, H, Hkv, D, bs, B, MB, NB, max_query_len, dtype, err, stream)
    a = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 8, 8, 128, 16, 4, 8, 100, 64, 2, None, None]

    def rc(**kw):
        b = list(a)
        for i, v in kw.items():
            b[int(i[1:])] = v
        return L.pkv_paged_attention_prefill(*b)
    assert rc(a12=0) == OK and rc(a15=0) == OK       # nothing to do
    assert rc(a15=-1) == INV
    assert rc(a6=None) == INV and rc(a6=FAKE + 2) == INV
    assert rc(a16=0) == UNS                          # binary32: no tensor-core path
    assert rc(a10=96) == UNS and rc(a11=64) == UNS
    assert rc(a9=3) == INV                           # 8 % 3 != 0
    assert rc(a1=FAKE + 8) == INV


def test_no_fallback_without_library(tmp_path):
    """A copy of the binding without its compiled library refuses to import."""
    import shutil
    pkg = tmp_path / "paged_kv_cache_204_gb300"
    shutil.copytree(os.path.join(ROOT, "paged_kv_cache_204_gb300"), pkg,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    code = ("import sys\n"
            f"sys.path.insert(0, {str(tmp_path)!r})\n"
            "try:\n"
            "    import paged_kv_cache_204_gb300\n"
            "    print('imported')\n"
            "except ImportError as e:\n"
            "    print('ImportError', e)\n")
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True)
    assert "ImportError" in r.stdout and "missing" in r.stdout, r.stdout + r.stderr
