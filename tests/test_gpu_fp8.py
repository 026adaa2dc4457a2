"""fp8 (E4M3) KV cache on the GPU against the oracle.

"Efficient Memory Management for Large Language Model Serving with
PagedAttention" (hackerpapers page), section "In the conversation":
quantising the KV cache cuts its memory footprint. The cache write must
produce exactly the oracle's codes (the rounding decision is taken on the
same binary32 quotient on both sides); block copies are byte copies; decode
attention over the codes must match the oracle's fp64 attention over the
decoded, scaled values within the tolerance of the 16-bit paths."""
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


def finite_codes(rng, shape) -> np.ndarray:
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7f) == 0x7f, c ^ 0x01, c).astype(np.uint8)  # no NaN codes


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 8), (128, 32)])
def test_fp8_cache_write_bit_exact(dtype, D, bs):
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(400 + D + bs)
    T, Hkv, NB = 300, 4, 64
    # values spread so that some quotients saturate and many are subnormal
    k = H.round_to_storage(rng.standard_normal((T, Hkv, D)) * np.exp(rng.uniform(-8, 3, (T, Hkv, D))), dtype)
    v = H.round_to_storage(rng.standard_normal((T, Hkv, D)), dtype)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::17] = -1
    kc = rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ks, vs = 0.037, 0.011
    pkv.reshape_and_cache_fp8(up16(k, dtype), up16(v, dtype), gk, gv, torch.from_numpy(slots).to(DEV), ks, vs,
                              dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oracle.reshape_and_cache_fp8(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D, block_size=bs, src_dtype=dtype,
                                 k_scale=ks, v_scale=vs)
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)
    assert (kc == 0x7e).any() or (kc == 0xfe).any()  # saturation was exercised


def test_fp8_copy_blocks_bit_exact():
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(41)
    NB, Hkv, bs, D = 40, 4, 16, 128
    kc = rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:10], perm[10:20]], 1).astype(np.int64)
    gk, gv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    pkv.copy_blocks(gk, gv, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    oracle.copy_blocks(kc.view(np.uint16), vc.view(np.uint16), pairs, num_kv_heads=Hkv, head_dim=D // 2,
                       block_size=bs, dtype="f16")  # byte copy of the same blocks
    assert np.array_equal(gk.cpu().numpy(), kc) and np.array_equal(gv.cpu().numpy(), vc)


CASES = [
    # (q dtype, H, Hkv, D, bs, lengths)
    ("f16", 8, 8, 128, 16, [1, 17, 300, 2048, 777, 16]),
    ("bf16", 8, 2, 64, 8, [5, 129, 1500, 40]),
    ("f16", 8, 2, 128, 32, [3000, 1, 64, 333]),
    ("bf16", 4, 1, 128, 16, [2500, 2500, 7]),
    ("f16", 4, 4, 64, 16, [0, 9, 1000]),
    # one query head per kv head (the tensor-core tile): bf16 queries, small
    # and large blocks, ragged last tiles
    ("bf16", 8, 8, 64, 8, [5, 129, 1500, 40]),
    ("bf16", 4, 4, 128, 32, [2500, 31, 33, 1, 64]),
]


@pytest.mark.parametrize("qd,H_,Hkv,D,bs,lens", CASES, ids=[f"{c[0]}-h{c[1]}/{c[2]}-d{c[3]}-bs{c[4]}" for c in CASES])
def test_fp8_decode_matches_oracle(qd, H_, Hkv, D, bs, lens):
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(sum(lens) + D + bs)
    lens = np.asarray(lens, dtype=np.int32)
    B = lens.size
    MB = max(1, int(-(-lens.max() // bs)))
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + 11
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    kc = finite_codes(rng, (NB, Hkv, bs, D))
    vc = finite_codes(rng, (NB, Hkv, bs, D))
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), qd)
    scale, ks, vs = 1.0 / np.sqrt(D), 0.0123, 0.0311
    out = torch.empty((B, H_, D), dtype=TD[qd], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    args = (up16(q, qd), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV), torch.from_numpy(bt).to(DEV),
            torch.from_numpy(lens).to(DEV))
    for rep in range(2):  # the workspace is reused: its counters must come back zero
        pkv.paged_attention_decode_fp8(out, *args, scale, ks, vs, mcl, workspace=ws, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle.paged_attention_fp8(q, kc, vc, bt, lens, scale=scale, k_scale=ks, v_scale=vs, num_heads=H_,
                                         num_kv_heads=Hkv, head_dim=D, block_size=bs, q_dtype=qd, threads=8)
        assert_close(to_f64(out), ref, f"fp8 decode rep {rep}")


@pytest.mark.parametrize("qd,D", [("bf16", 128), ("f16", 128), ("bf16", 64)])
def test_fp8_decode_poison_and_query_range(qd, D):
    """Every cache byte outside the sequences' tokens is a NaN code (0x7f or
    0xff), so a kernel that lets a masked key or value reach the arithmetic
    gives NaN. Query rows span 2^-20 .. 2^20 times N(0, 1) (bf16) or
    2^-8 .. 2^8 (f16), so a query path that loses range or precision on the
    way into 16-bit operands shows up against the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(4099 + D)
    H_, bs = 6, 16
    lens = np.asarray([1, 15, 16, 17, 31, 32, 33, 700, 0, 95], dtype=np.int32)
    B = lens.size
    MB = max(1, int(-(-lens.max() // bs)))
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + 5
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    kc = np.where(rng.random((NB, H_, bs, D)) < 0.5, 0x7f, 0xff).astype(np.uint8)
    vc = np.where(rng.random((NB, H_, bs, D)) < 0.5, 0x7f, 0xff).astype(np.uint8)
    k = 0
    for s in range(B):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        for j in range(nblk[s]):
            n = min(bs, int(lens[s]) - j * bs)
            kc[bt[s, j], :, :n] = finite_codes(rng, (H_, n, D))
            vc[bt[s, j], :, :n] = finite_codes(rng, (H_, n, D))
        k += nblk[s]
    span = 20 if qd == "bf16" else 8
    row_scale = np.exp2(rng.integers(-span, span + 1, size=(B, H_, 1)).astype(np.float64))
    q = rng.standard_normal((B, H_, D)) * row_scale
    q[0, 0, 0] *= 2.0**(span if qd == "bf16" else 4)  # one element far above the rest of its row
    q = H.round_to_storage(q, qd)
    scale, ks, vs = 1.0 / np.sqrt(D), 0.0123, 0.0311
    out = torch.empty((B, H_, D), dtype=TD[qd], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    pkv.paged_attention_decode_fp8(out, up16(q, qd), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                                   torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV), scale, ks, vs, mcl,
                                   workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_f64(out)
    assert np.isfinite(got).all()
    ref = oracle.paged_attention_fp8(q, kc, vc, bt, lens, scale=scale, k_scale=ks, v_scale=vs, num_heads=H_,
                                     num_kv_heads=H_, head_dim=D, block_size=bs, q_dtype=qd, threads=8)
    assert_close(got, ref, "fp8 decode, poison and query range")


def test_fp8_decode_full_size_sampled():
    """LLaMA-13B-shaped step (128 sequences x 40 heads, lognormal lengths) with
    fp8 caches: every output row of 12 sampled sequences against the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    import synth
    cfg = synth.get("llama13b")
    st = synth.build(cfg)
    rng = np.random.default_rng(43)
    B, H_, Hkv, D, bs = st.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    used = np.unique(st.block_tables[st.block_tables >= 0])
    NB = int(used.max()) + 1
    kc = torch.empty((NB, Hkv, bs, D), dtype=torch.uint8, device=DEV)
    vc = torch.empty_like(kc)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(44)
    kc.copy_(torch.randint(0, 0x7e, kc.shape, generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8))
    vc.copy_(torch.randint(0, 0x7e, vc.shape, generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8))
    sign = torch.randint(0, 2, kc.shape, generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8) << 7
    kc |= sign
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), "bf16")
    out = torch.empty((B, H_, D), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = pkv.new_workspace(B, H_, D, st.max_context_len, device=DEV)
    bt_d, cl_d = torch.from_numpy(st.block_tables).to(DEV), torch.from_numpy(st.context_lens).to(DEV)
    pkv.paged_attention_decode_fp8(out, up16(q, "bf16"), kc, vc, bt_d, cl_d, cfg.scale, 0.02, 0.05,
                                   st.max_context_len, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    seqs = np.sort(rng.choice(B, 12, replace=False))
    sub_bt = st.block_tables[seqs]
    ids = np.unique(sub_bt[sub_bt >= 0])
    remap = np.full(NB, -1, dtype=np.int32)
    remap[ids] = np.arange(ids.size, dtype=np.int32)
    bt_c = np.where(sub_bt >= 0, remap[np.maximum(sub_bt, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(ids.astype(np.int64)).to(DEV)
    ref = oracle.paged_attention_fp8(q[seqs], kc[idx].cpu().numpy(), vc[idx].cpu().numpy(), bt_c,
                                     st.context_lens[seqs], scale=cfg.scale, k_scale=0.02, v_scale=0.05,
                                     num_heads=H_, num_kv_heads=Hkv, head_dim=D, block_size=bs, q_dtype="bf16",
                                     threads=8)
    assert_close(to_f64(out)[seqs], ref, "fp8 full-size sampled")


def test_fp8_decode_wait_timeout_is_reported_and_context_survives():
    """The tensor-core fp8 tile (one query head per kv head, TMA loads at head
    dim 128) under a wait limit of 0: PKV_DEV_ERR_TIMEOUT and nothing else,
    then a call with the default limit (workspace cleared) matches the oracle."""
    import paged_kv_cache_204_gb300 as pkv
    rng = np.random.default_rng(4242)
    H_, D, bs = 8, 128, 16
    lens = np.asarray([700, 33, 1200, 5, 64, 900], dtype=np.int32)
    B = lens.size
    MB = int(-(-lens.max() // bs))
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    kc = finite_codes(rng, (NB, H_, bs, D))
    vc = finite_codes(rng, (NB, H_, bs, D))
    q = H.round_to_storage(rng.standard_normal((B, H_, D)), "bf16")
    scale, ks, vs = 1.0 / np.sqrt(D), 0.02, 0.03
    out = torch.empty((B, H_, D), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mcl = int(lens.max())
    ws = pkv.new_workspace(B, H_, D, mcl, device=DEV)
    args = (up16(q, "bf16"), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
            torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV))
    old = pkv.get_wait_timeout_ns()
    try:
        pkv.set_wait_timeout_ns(0)
        pkv.paged_attention_decode_fp8(out, *args, scale, ks, vs, mcl, workspace=ws, dev_err=err)
        torch.cuda.synchronize()
        code = int(err.item())
    finally:
        pkv.set_wait_timeout_ns(old)
    assert code & pkv.DEV_ERR_TIMEOUT
    assert code & ~pkv.DEV_ERR_TIMEOUT == 0
    err.zero_()
    ws.zero_()
    pkv.paged_attention_decode_fp8(out, *args, scale, ks, vs, mcl, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_attention_fp8(q, kc, vc, bt, lens, scale=scale, k_scale=ks, v_scale=vs, num_heads=H_,
                                     num_kv_heads=H_, head_dim=D, block_size=bs, q_dtype="bf16", threads=8)
    assert_close(to_f64(out), ref, "fp8 decode after timeout")
