"""4-bit (q4_0) KV cache on the GPU against the oracle.

"Efficient Memory Management for Large Language Model Serving with
PagedAttention" (hackerpapers page), section "In the conversation": 4-bit
KV-cache quantisation (the q4_0 cache type) cuts the cache to about a
quarter. The cache write must produce exactly the oracle's bytes (every
rounding decision is taken in binary32 on both sides); block copies are
byte copies; decode attention over q4_0 rows must match the oracle's fp64
attention over the values d (q - 8) within the tolerance of the 16-bit paths."""
import numpy as np
import pytest
import torch

import oracle
import synth.host as H
from gpu_helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}
DEV = torch.device("cuda", 0)


def up16(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(TD[dtype])


def q4_pool(rng, NB, Hkv, bs, D, scale_sigma) -> np.ndarray:
    """Random q4_0 rows: any code bytes, finite binary16 scales."""
    rb = oracle.q4_0_row_bytes(D)
    p = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
    sc = (rng.standard_normal((NB, Hkv, bs, D // 32)) * scale_sigma).astype(np.float16)
    p[..., :D // 16] = sc.view(np.uint8).reshape(NB, Hkv, bs, D // 16)
    return p


def paged_tables(rng, lens, bs, extra=7):
    lens = np.asarray(lens, dtype=np.int32)
    B = lens.size
    MB = max(1, int(-(-lens.max() // bs)))
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + extra
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    return lens, bt, NB, nblk


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 8), (128, 32)])
def test_q4_cache_write_bit_exact(dtype, D, bs):
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(500 + D + bs)
    T, Hkv, NB = 300, 4, 64
    rb = oracle.q4_0_row_bytes(D)
    # magnitudes over many binades (tiny scales round to binary16 subnormals)
    raw = rng.standard_normal((T, Hkv, D)) * np.exp(rng.uniform(-14, 3, (T, Hkv, 1)))
    raw[5, 1, :32] = 0.0                     # a zero block
    raw[6, 0, :32] = 0.25                    # magnitude ties of both signs
    raw[6, 0, 3], raw[6, 0, 9] = -2.0, 2.0
    raw[7, 2] = np.round(raw[7, 2] * 8) / 8  # many exact products
    if dtype == "bf16":
        raw[8, 3, 32:64] *= 1e7              # a scale beyond binary16: infinite
    k = H.round_to_storage(raw, dtype)
    v = H.round_to_storage(rng.standard_normal((T, Hkv, D)), dtype)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::17] = -1
    kc = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.reshape_and_cache_q4_0(up16(k, dtype), up16(v, dtype), gk, gv, torch.from_numpy(slots).to(DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oracle.reshape_and_cache_q4_0(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D, block_size=bs, src_dtype=dtype)
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)


def test_q4_cache_write_bad_slot_is_reported():
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(51)
    T, Hkv, D, bs, NB = 5, 2, 128, 16, 4
    rb = oracle.q4_0_row_bytes(D)
    k = H.round_to_storage(rng.standard_normal((T, Hkv, D)), "f16")
    slots = np.array([0, 5, NB * bs + 1, -1, 63], dtype=np.int64)
    kc = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(kc.copy()).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.reshape_and_cache_q4_0(up16(k, "f16"), up16(k, "f16"), gk, gv, torch.from_numpy(slots).to(DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_ERR_SLOT
    ek = kc.copy()
    bad = oracle.reshape_and_cache_q4_0(k, k, ek, kc.copy(), slots, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                        src_dtype="f16")
    assert bad == 1 and np.array_equal(gk.cpu().numpy(), ek)


def test_q4_copy_blocks_bit_exact():
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(53)
    NB, Hkv, bs, D = 40, 4, 16, 128
    kc = q4_pool(rng, NB, Hkv, bs, D, 0.05)
    vc = q4_pool(rng, NB, Hkv, bs, D, 0.05)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:10], perm[10:20]], 1).astype(np.int64)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    pkv.copy_blocks_q4_0(gk, gv, torch.from_numpy(pairs).to(DEV), D)
    torch.cuda.synchronize()
    ek, ev = kc.copy(), vc.copy()
    for s, d in pairs:
        ek[d], ev[d] = kc[s], vc[s]
    assert np.array_equal(gk.cpu().numpy(), ek) and np.array_equal(gv.cpu().numpy(), ev)


CASES = [
    # (q dtype, H, Hkv, D, bs, lengths)
    ("f16", 8, 8, 128, 16, [1, 17, 300, 2048, 777, 16]),
    ("bf16", 8, 8, 64, 8, [5, 129, 1500, 40]),
    ("f16", 8, 2, 128, 32, [3000, 1, 64, 333]),
    ("bf16", 4, 1, 128, 16, [2500, 2500, 7]),
    ("f16", 4, 4, 64, 16, [0, 9, 1000]),
    ("bf16", 4, 4, 128, 32, [2500, 31, 33, 1, 64]),
]


@pytest.mark.parametrize("qd,H_,Hkv,D,bs,lens", CASES, ids=[f"{c[0]}-h{c[1]}/{c[2]}-d{c[3]}-bs{c[4]}" for c in CASES])
def test_q4_decode_matches_oracle(qd, H_, Hkv, D, bs, lens):
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(sum(lens) + D + bs + 7)
    lens, bt, NB, _ = paged_tables(rng, lens, bs)
    B = lens.size
    kc = q4_pool(rng, NB, Hkv, bs, D, 0.03)
    vc = q4_pool(rng, NB, Hkv, bs, D, 0.1)
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), qd)
    scale = 1.0 / np.sqrt(D)
    out = torch.empty((B, H_, D), dtype=TD[qd], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    args = (up16(q, qd), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV), torch.from_numpy(bt).to(DEV),
            torch.from_numpy(lens).to(DEV))
    ref = oracle.paged_attention_q4_0(q, kc, vc, bt, lens, scale=scale, num_heads=H_, num_kv_heads=Hkv, head_dim=D,
                                      block_size=bs, q_dtype=qd, threads=8)
    for rep in range(2):  # the workspace is reused: its counters must come back zero
        pkv.paged_attention_decode_q4_0(out, *args, scale, mcl, workspace=ws, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(to_f64(out), ref, f"q4_0 decode rep {rep}")


@pytest.mark.parametrize("qd,D", [("bf16", 128), ("f16", 128), ("bf16", 64)])
def test_q4_decode_poison_and_query_range(qd, D):
    """Every cache row outside the sequences' tokens has NaN or infinite
    scales, so a kernel that lets a masked key or value reach the arithmetic
    gives NaN. Query rows span 2^-20 .. 2^20 (bf16) or 2^-8 .. 2^8 (f16)
    times N(0, 1), so a query path that loses range or precision on the way
    into 16-bit operands shows up against the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(5099 + D)
    H_, bs = 6, 16
    lens, bt, NB, nblk = paged_tables(rng, [1, 15, 16, 17, 31, 32, 33, 700, 0, 95], bs, extra=5)
    B = lens.size
    rb = oracle.q4_0_row_bytes(D)
    kc = rng.integers(0, 256, (NB, H_, bs, rb), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, H_, bs, rb), dtype=np.uint8)
    bad_scales = np.where(rng.random((NB, H_, bs, D // 32)) < 0.5, 0x7e00, 0xfc00).astype(np.uint16)
    kc[..., :D // 16] = bad_scales.view(np.uint8).reshape(NB, H_, bs, D // 16)
    vc[..., :D // 16] = bad_scales[::-1].view(np.uint8).reshape(NB, H_, bs, D // 16)
    good_k, good_v = q4_pool(rng, NB, H_, bs, D, 0.03), q4_pool(rng, NB, H_, bs, D, 0.1)
    for s in range(B):
        for j in range(nblk[s]):
            n = min(bs, int(lens[s]) - j * bs)
            kc[bt[s, j], :, :n] = good_k[bt[s, j], :, :n]
            vc[bt[s, j], :, :n] = good_v[bt[s, j], :, :n]
    span = 20 if qd == "bf16" else 8
    row_scale = np.exp2(rng.integers(-span, span + 1, size=(B, H_, 1)).astype(np.float64))
    q = rng.standard_normal((B, H_, D)) * row_scale
    q[0, 0, 0] *= 2.0**(span if qd == "bf16" else 4)
    q = H.round_to_storage(q, qd)
    scale = 1.0 / np.sqrt(D)
    out = torch.empty((B, H_, D), dtype=TD[qd], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    pkv.paged_attention_decode_q4_0(out, up16(q, qd), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                                    torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV), scale, mcl,
                                    workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_f64(out)
    assert np.isfinite(got).all()
    ref = oracle.paged_attention_q4_0(q, kc, vc, bt, lens, scale=scale, num_heads=H_, num_kv_heads=H_, head_dim=D,
                                      block_size=bs, q_dtype=qd, threads=8)
    assert_close(got, ref, "q4_0 decode, poison and query range")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_q4_write_then_decode_end_to_end(dtype):
    """The whole q4_0 path through the C ABI: rows written by the cache write
    kernel, then decoded; against the oracle's own write and attention."""
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(57 if dtype == "f16" else 58)
    H_, Hkv, D, bs = 8, 4, 128, 16
    lens, bt, NB, nblk = paged_tables(rng, [40, 1, 513, 200, 17], bs, extra=3)
    B = lens.size
    rb = oracle.q4_0_row_bytes(D)
    slots, rows = [], []
    for s in range(B):
        for t in range(int(lens[s])):
            slots.append(int(bt[s, t // bs]) * bs + t % bs)
    T = len(slots)
    k = H.round_to_storage(rng.standard_normal((T, Hkv, D)) * 0.5, dtype)
    v = H.round_to_storage(rng.standard_normal((T, Hkv, D)), dtype)
    slots = np.asarray(slots, dtype=np.int64)
    kc = np.zeros((NB, Hkv, bs, rb), dtype=np.uint8)
    vc = np.zeros_like(kc)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.reshape_and_cache_q4_0(up16(k, dtype), up16(v, dtype), gk, gv, torch.from_numpy(slots).to(DEV), dev_err=err)
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), dtype)
    out = torch.empty((B, H_, D), dtype=TD[dtype], device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    pkv.paged_attention_decode_q4_0(out, up16(q, dtype), gk, gv, torch.from_numpy(bt).to(DEV),
                                    torch.from_numpy(lens).to(DEV), 1.0 / np.sqrt(D), mcl, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oracle.reshape_and_cache_q4_0(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D, block_size=bs, src_dtype=dtype)
    assert np.array_equal(gk.cpu().numpy(), kc) and np.array_equal(gv.cpu().numpy(), vc)
    ref = oracle.paged_attention_q4_0(q, kc, vc, bt, lens, scale=1.0 / np.sqrt(D), num_heads=H_, num_kv_heads=Hkv,
                                      head_dim=D, block_size=bs, q_dtype=dtype, threads=8)
    assert_close(to_f64(out), ref, "q4_0 write + decode")


def test_q4_decode_full_size_sampled():
    """LLaMA-13B-shaped step (128 sequences x 40 heads, lognormal lengths) with
    q4_0 caches: every output row of 12 sampled sequences against the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    import synth
    cfg = synth.get("llama13b")
    st = synth.build(cfg)
    rng = np.random.default_rng(59)
    B, H_, Hkv, D, bs = st.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    used = np.unique(st.block_tables[st.block_tables >= 0])
    NB = int(used.max()) + 1
    rb = oracle.q4_0_row_bytes(D)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(60)

    def pool(sigma):
        p = torch.randint(0, 256, (NB, Hkv, bs, rb), generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8)
        sc = (torch.randn((NB, Hkv, bs, D // 32), generator=gen, device=DEV) * sigma).to(torch.float16)
        p[..., :D // 16] = sc.view(torch.uint8).reshape(NB, Hkv, bs, D // 16)
        return p

    kc, vc = pool(0.03), pool(0.1)
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), "bf16")
    out = torch.empty((B, H_, D), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = pkv.new_workspace(B, H_, D, st.max_context_len, device=DEV)
    bt_d, cl_d = torch.from_numpy(st.block_tables).to(DEV), torch.from_numpy(st.context_lens).to(DEV)
    pkv.paged_attention_decode_q4_0(out, up16(q, "bf16"), kc, vc, bt_d, cl_d, cfg.scale, st.max_context_len,
                                    workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    seqs = np.sort(rng.choice(B, 12, replace=False))
    sub_bt = st.block_tables[seqs]
    ids = np.unique(sub_bt[sub_bt >= 0])
    remap = np.full(NB, -1, dtype=np.int32)
    remap[ids] = np.arange(ids.size, dtype=np.int32)
    bt_c = np.where(sub_bt >= 0, remap[np.maximum(sub_bt, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(ids.astype(np.int64)).to(DEV)
    ref = oracle.paged_attention_q4_0(q[seqs], kc[idx].cpu().numpy(), vc[idx].cpu().numpy(), bt_c,
                                      st.context_lens[seqs], scale=cfg.scale, num_heads=H_, num_kv_heads=Hkv,
                                      head_dim=D, block_size=bs, q_dtype="bf16", threads=8)
    assert_close(to_f64(out)[seqs], ref, "q4_0 full-size sampled")


def test_q4_decode_wait_timeout_is_reported_and_context_survives():
    """Under a wait limit of 0: PKV_DEV_ERR_TIMEOUT and nothing else; then a
    call with the default limit (workspace cleared) matches the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(5242)
    H_, D, bs = 8, 128, 16
    lens, bt, NB, _ = paged_tables(rng, [700, 33, 1200, 5, 64, 900], bs, extra=3)
    B = lens.size
    kc = q4_pool(rng, NB, H_, bs, D, 0.03)
    vc = q4_pool(rng, NB, H_, bs, D, 0.1)
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), "bf16")
    scale = 1.0 / np.sqrt(D)
    out = torch.empty((B, H_, D), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    args = (up16(q, "bf16"), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
            torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV))
    old = pkv.get_wait_timeout_ns()
    try:
        pkv.set_wait_timeout_ns(0)
        pkv.paged_attention_decode_q4_0(out, *args, scale, mcl, workspace=ws, dev_err=err)
        torch.cuda.synchronize()
        code = int(err.item())
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT
    assert code & ~pkv.DEV_ERR_TIMEOUT == 0
    err.zero_()
    ws.zero_()
    pkv.paged_attention_decode_q4_0(out, *args, scale, mcl, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_attention_q4_0(q, kc, vc, bt, lens, scale=scale, num_heads=H_, num_kv_heads=H_, head_dim=D,
                                      block_size=bs, q_dtype="bf16", threads=8)
    assert_close(to_f64(out), ref, "q4_0 decode after timeout")
