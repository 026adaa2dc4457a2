"""Checks that pin the oracle to facts other than itself.

Each pin takes an oracle build `L` (None = the default build) and raises
AssertionError when the oracle disagrees with:
  - the storage formats' definitions (element decoders vs numpy's binary16 and
    the bfloat16 = upper-half-of-binary32 definition);
  - closed forms of softmax attention (context 1 returns V; a zero query or
    identical keys average V; one dominant logit selects its V; two tokens
    reduce to the logistic function; grouped heads read kv head h // group);
  - high-precision brute force (mpmath, 200-bit) on tiny inputs;
  - the paging facts of "PagedAttention: the KV cache was the bottleneck all
    along", section "Virtual memory for attention": the block table only says
    where a token lives (paged == dense over the same tokens; any physical
    permutation gives identical bits), and copy-on-write sharing gives the
    same result as private copies;
  - the log-sum-exp combination of split contexts;
  - byte-level placement of cache writes and block copies, checked with numpy
    indexing of the [num_blocks][kv_heads][block_size][head_dim] layout;
  - paged prefill (causal queries of a sequence's last tokens): one query
    per sequence is decode; each query equals dense attention over exactly
    its own prefix, gathered by numpy indexing;
  - the fp8 (E4M3) cache: the code table and round-to-nearest-even of
    PyTorch's float8_e4m3fn conversion (a library routine), saturation at
    448, ties to the even code, and attention over E4M3 pools equal bit for
    bit to the binary32 oracle over the exactly decoded values;
  - the 4-bit (q4_0) cache: the binary16 rounding of the scale against
    numpy's conversion, exact blocks d (k - 8) whose codes are known, the
    hand-derived rules (first maximum, rounding half up, the clamp at 15,
    the zero block), the error bound of the format, byte placement of the
    cache write, and attention over q4_0 pools equal bit for bit to the
    binary32 oracle over the values numpy reads back from the rows.

tests/test_oracle_pins.py runs them on the oracle; tests/test_oracle_mutations.py
runs them on copies with planted mistakes and expects each copy to fail one.
"""
from __future__ import annotations

import numpy as np
import scipy.special

import oracle
import synth
import synth.host as H

DTYPES = ("f32", "f16", "bf16")


def _rand_store(rng, shape, dtype, scale=1.0):
    return H.round_to_storage(rng.standard_normal(shape) * scale, dtype)


def _dec(a, dtype):
    """Reference decode with numpy (not the oracle's decoders)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype, q_scale=1.0):
    """Random q and pools; each sequence gets distinct random blocks; rows past
    a sequence's length are poison."""
    lens = np.asarray(lens, dtype=np.int32)
    MB = max(1, int(-(-lens.max() // bs)))
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        n = -(-int(lens[s]) // bs)
        bt[s, :n] = perm[k:k + n]
        k += n
    assert k <= NB
    kc = H.poison((NB, Hkv, bs, D), dtype)
    vc = H.poison((NB, Hkv, bs, D), dtype)
    for s in range(B):
        for t in range(int(lens[s])):
            p = bt[s, t // bs]
            kc[p, :, t % bs, :] = _rand_store(rng, (Hkv, D), dtype)
            vc[p, :, t % bs, :] = _rand_store(rng, (Hkv, D), dtype)
    q = _rand_store(rng, (B, H_, D), dtype, q_scale)
    return q, kc, vc, bt, lens


def _attn(L, q, kc, vc, bt, lens, H_, Hkv, D, bs, dtype, scale):
    return oracle.paged_attention(q, kc, vc, bt, lens, scale=scale, num_heads=H_,
                                  num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dtype, L=L)


def _gather_dense(kc, bt, lens, bs):
    """Each sequence's rows, in token order, by numpy indexing of the layout."""
    rows = []
    for s in range(len(lens)):
        t = np.arange(int(lens[s]))
        rows.append(kc[bt[s, t // bs], :, t % bs, :])
    return np.ascontiguousarray(np.concatenate(rows, axis=0)) if rows else kc[:0, :, 0, :]


# ---------------------------------------------------------------- decoders
@np.errstate(invalid="ignore")
def pin_decoders(L=None):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_elements(bits, "f16", L)
    assert np.array_equal(got, bits.view(np.float16).astype(np.float64), equal_nan=True), "f16 decode"
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.decode_elements(bits, "bf16", L)
    assert np.array_equal(got, ref, equal_nan=True), "bf16 decode"
    rng = np.random.default_rng(7)
    u = np.concatenate([rng.integers(0, 2 ** 32, 50000, dtype=np.uint64).astype(np.uint32),
                        np.array([0, 1, 0x7FFFFF, 0x800000, 0x7F7FFFFF, 0x7F800000, 0xFF800000,
                                  0x80000001, 0x3F800000], dtype=np.uint32)])
    got = oracle.decode_elements(u.view(np.float32), "f32", L)
    assert np.array_equal(got, u.view(np.float32).astype(np.float64), equal_nan=True), "f32 decode"


# ---------------------------------------------------------------- closed forms
def pin_context_one(L=None):
    """A context of one token returns that token's V row exactly."""
    rng = np.random.default_rng(11)
    for dtype in DTYPES:
        B, H_, Hkv, D, bs, NB = 5, 4, 2, 64, 8, 16
        q, kc, vc, bt, lens = _random_paged(rng, B, H_, Hkv, D, bs, NB, [1] * B, dtype)
        out = _attn(L, q, kc, vc, bt, lens, H_, Hkv, D, bs, dtype, 0.3)
        for s in range(B):
            for h in range(H_):
                assert np.array_equal(out[s, h], _dec(vc[bt[s, 0], h // 2, 0], dtype)), \
                    f"context 1 {dtype} s={s} h={h}"


def pin_uniform_weights(L=None):
    """q = 0, or all keys of a head equal: every weight is the same, so the
    output is the mean of the V rows."""
    rng = np.random.default_rng(12)
    B, H_, Hkv, D, bs, NB = 4, 2, 2, 64, 16, 40
    lens = [37, 1, 64, 100]
    for dtype in DTYPES:
        q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype)
        q0 = np.zeros_like(q)
        out = _attn(L, q0, kc, vc, bt, lens_, H_, Hkv, D, bs, dtype, 0.125)
        kq = kc.copy()
        for s in range(B):  # identical keys within each (sequence, head)
            for t in range(lens[s]):
                kq[bt[s, t // bs], :, t % bs, :] = kc[bt[s, 0], :, 0, :]
        out2 = _attn(L, q, kq, vc, bt, lens_, H_, Hkv, D, bs, dtype, 0.125)
        for s in range(B):
            t = np.arange(lens[s])
            mean = _dec(vc[bt[s, t // bs], :, t % bs, :], dtype).mean(axis=0)  # [Hkv, D]
            assert np.allclose(out[s], mean, rtol=0, atol=1e-12), f"q=0 mean {dtype}"
            assert np.allclose(out2[s], mean, rtol=0, atol=1e-12), f"equal keys mean {dtype}"


def pin_dominant_logit(L=None):
    """One logit 80 above all others (weights e^-80 elsewhere): the output is
    that token's V to within 1e-30 relative."""
    rng = np.random.default_rng(13)
    B, H_, Hkv, D, bs, NB = 3, 1, 1, 64, 16, 30
    lens = [50, 50, 50]
    q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, "f32")
    q[:] = 0.0
    q[:, :, 0] = 1.0
    for s, star in enumerate((0, 23, 49)):
        for t in range(50):
            kc[bt[s, t // bs], 0, t % bs, :] = 0.0
        kc[bt[s, star // bs], 0, star % bs, 0] = 80.0
    out = _attn(L, q, kc, vc, bt, lens_, H_, Hkv, D, bs, "f32", 1.0)
    for s, star in enumerate((0, 23, 49)):
        v = _dec(vc[bt[s, star // bs], 0, star % bs], "f32")
        assert np.allclose(out[s, 0], v, rtol=1e-25, atol=1e-30), f"dominant logit s={s}"


def pin_two_tokens(L=None):
    """Softmax over two tokens is the logistic function of the logit gap:
    out = (1 - w) V0 + w V1 with w = expit(scale * q.(k1 - k0)). Tokens sit in
    different physical blocks (block_size 1)."""
    for scale, a, b0, b1 in ((0.125, 3.0, 2.0, -5.0), (0.5, -1.5, 4.0, 0.25), (1.0, 0.0, 1.0, 9.0)):
        D, NB = 64, 7
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, 5] = a
        kc = H.poison((NB, 1, 1, D), "f32")
        vc = H.poison((NB, 1, 1, D), "f32")
        bt = np.array([[4, 2]], np.int32)
        kc[4, 0, 0, :] = 0.0
        kc[2, 0, 0, :] = 0.0
        kc[4, 0, 0, 5] = b0
        kc[2, 0, 0, 5] = b1
        rng = np.random.default_rng(14)
        vc[4, 0, 0, :] = rng.standard_normal(D).astype(np.float32)
        vc[2, 0, 0, :] = rng.standard_normal(D).astype(np.float32)
        out = _attn(L, q, kc, vc, bt, np.array([2], np.int32), 1, 1, D, 1, "f32", scale)
        w = scipy.special.expit(scale * a * (b1 - b0))
        ref = (1 - w) * vc[4, 0, 0].astype(np.float64) + w * vc[2, 0, 0].astype(np.float64)
        assert np.allclose(out[0, 0], ref, rtol=1e-14, atol=1e-15), f"two tokens scale={scale}"


def pin_gqa_mapping(L=None):
    """Grouped heads: query head h reads kv head h // (H / Hkv). With V of kv
    head g equal to the constant 2^(g-1) everywhere, every output element of
    head h is exactly 2^(h//group - 1)."""
    rng = np.random.default_rng(15)
    B, H_, Hkv, D, bs, NB = 3, 6, 3, 64, 8, 24
    for dtype in DTYPES:
        q, kc, vc, bt, lens = _random_paged(rng, B, H_, Hkv, D, bs, NB, [9, 17, 30], dtype)
        for g in range(Hkv):
            c = H.round_to_storage(np.array(2.0 ** (g - 1)), dtype)
            used = vc[:, g][~H.is_poison(vc[:, g])]
            vc[:, g][~H.is_poison(vc[:, g])] = c
            assert used.size
        out = _attn(L, q, kc, vc, bt, lens, H_, Hkv, D, bs, dtype, 0.2)
        for h in range(H_):
            assert np.all(out[:, h, :] == 2.0 ** (h // 2 - 1)), f"gqa head {h} {dtype}"


# ---------------------------------------------------------------- brute force
def pin_brute_force(L=None):
    """Tiny inputs against 200-bit mpmath evaluation of the definition."""
    import mpmath
    mpmath.mp.prec = 200
    rng = np.random.default_rng(16)
    for dtype in DTYPES:
        B, H_, Hkv, D, bs, NB = 3, 2, 1, 4, 2, 12
        lens = [1, 4, 5]
        q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype)
        scale = 0.7
        out = _attn(L, q, kc, vc, bt, lens_, H_, Hkv, D, bs, dtype, scale)
        for s in range(B):
            for h in range(H_):
                qs = [mpmath.mpf(float(x)) for x in _dec(q[s, h], dtype)]
                xs, vs = [], []
                for t in range(lens[s]):
                    p, r = bt[s, t // bs], t % bs
                    kr = _dec(kc[p, 0, r], dtype)
                    xs.append(mpmath.mpf(scale) * mpmath.fsum(qi * mpmath.mpf(float(ki))
                                                            for qi, ki in zip(qs, kr)))
                    vs.append(_dec(vc[p, 0, r], dtype))
                z = mpmath.fsum(mpmath.exp(x) for x in xs)
                for d in range(D):
                    ref = mpmath.fsum(mpmath.exp(x) * mpmath.mpf(float(v[d])) for x, v in zip(xs, vs)) / z
                    assert abs(float(ref) - out[s, h, d]) <= 1e-15 * (1 + abs(float(ref))), \
                        f"brute force {dtype} s={s} h={h} d={d}"


# ---------------------------------------------------------------- paging facts
def pin_dense_equivalence(L=None):
    """Paging only decides where token t lives: paged attention equals the same
    attention over the tokens laid out contiguously, bit for bit."""
    rng = np.random.default_rng(17)
    cases = [  # (B, H, Hkv, D, bs, NB, max_len, dtype)
        (4, 2, 2, 64, 16, 64, 100, "f32"),
        (5, 8, 2, 128, 8, 200, 150, "f16"),
        (3, 4, 4, 128, 32, 40, 300, "bf16"),
        (4, 6, 3, 64, 16, 80, 200, "f16"),
    ]
    for B, H_, Hkv, D, bs, NB, maxlen, dtype in cases:
        lens = rng.integers(1, maxlen + 1, B)
        q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype)
        scale = 1.0 / np.sqrt(D)
        out = _attn(L, q, kc, vc, bt, lens_, H_, Hkv, D, bs, dtype, scale)
        kd, vd = _gather_dense(kc, bt, lens_, bs), _gather_dense(vc, bt, lens_, bs)
        st = np.concatenate([[0], np.cumsum(lens_)]).astype(np.int64)
        ref = oracle.dense_attention(q, kd, vd, st, scale=scale, num_heads=H_, num_kv_heads=Hkv,
                                     head_dim=D, dtype=dtype, L=L)
        assert np.isfinite(out).all(), "poison reached the output"
        assert np.array_equal(out, ref), f"paged != dense {dtype} bs={bs}"


def pin_placement_invariance(L=None):
    """Any permutation of physical block ids (pool rows moved, tables
    renumbered) gives identical bits."""
    rng = np.random.default_rng(18)
    B, H_, Hkv, D, bs, NB = 6, 4, 2, 64, 8, 120
    for dtype in DTYPES:
        lens = rng.integers(1, 120, B)
        q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype)
        out = _attn(L, q, kc, vc, bt, lens_, H_, Hkv, D, bs, dtype, 0.1)
        perm = rng.permutation(NB)
        kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
        kc2[perm], vc2[perm] = kc, vc
        bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
        out2 = _attn(L, q, kc2, vc2, bt2, lens_, H_, Hkv, D, bs, dtype, 0.1)
        assert np.array_equal(out, out2), f"placement changed the result {dtype}"


def logical_streams(hw, hp):
    """Each served sequence's K and V rows in token order, built without the
    step's cache operations: prefix tokens from the pre-step pool through the
    pre-step tables, then the sequence's new rows. (This is what private,
    unshared copies of every sequence would hold.)"""
    st, cfg = hw.st, hw.cfg
    bs = cfg.block_size
    k0, v0 = hp.k_cache, hp.v_cache   # must be the pre-step pools
    ks, vs, lens = [], [], []
    for i, s in enumerate(hp.seqs):
        t = np.arange(int(st.prefix_lens[s]))
        p = hp.prefix_tables[i, t // bs]
        new = slice(int(st.new_start[s]), int(st.new_start[s + 1]))
        ks.append(np.concatenate([k0[p, :, t % bs, :], hw.new_k[new]], axis=0))
        vs.append(np.concatenate([v0[p, :, t % bs, :], hw.new_v[new]], axis=0))
        lens.append(ks[-1].shape[0])
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return np.ascontiguousarray(np.concatenate(ks)), np.ascontiguousarray(np.concatenate(vs)), start


def pin_copy_on_write(L=None):
    """Ref-counted sharing of prompt blocks + copy-on-write at divergence gives
    the same bits as every sample owning a private copy of its tokens; the
    step with new-token writes does the same for a plain batch."""
    for cfg, B in ((synth.get("cow").replace(num_heads=4, num_kv_heads=4, num_blocks=3000), 12),
                   (synth.get("cow").replace(num_heads=2, num_kv_heads=2, head_dim=64, block_size=8,
                                             dtype="bf16", num_blocks=3000), 9),
                   (synth.get("llama13b").replace(num_heads=4, num_kv_heads=2, num_blocks=2000), 10)):
        hw = H.generate(cfg, num_seqs=B)
        hp = H.compact_pools(hw)
        kd, vd, start = logical_streams(hw, hp)
        assert np.array_equal(start[1:] - start[:-1], hw.st.context_lens), "stream lengths"
        out, _, _ = oracle.decode_step(hp, hw, L=L)
        ref = oracle.dense_attention(hw.q, kd, vd, start, scale=cfg.scale, num_heads=cfg.num_heads,
                                     num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim,
                                     dtype=cfg.dtype, L=L)
        assert np.isfinite(out).all(), "poison reached the output"
        assert np.array_equal(out, ref), f"shared+CoW != private copies ({cfg.name})"


def pin_split_merge(L=None):
    """Chunked evaluation + log-sum-exp merge equals the single pass."""
    rng = np.random.default_rng(19)
    B, H_, Hkv, D, bs, NB = 4, 2, 1, 64, 16, 80
    for dtype in ("f32", "bf16"):
        lens = [1, 200, 333, 17]
        q, kc, vc, bt, lens_ = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype, q_scale=3.0)
        ref = _attn(L, q, kc, vc, bt, lens_, H_, Hkv, D, bs, dtype, 0.5)
        for chunk in (1, 3, 16, 64, 256, 4096):
            got = oracle.paged_attention_chunked(q, kc, vc, bt, lens_, scale=0.5, num_heads=H_,
                                                 num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                                 dtype=dtype, chunk=chunk, L=L)
            assert np.allclose(got, ref, rtol=1e-13, atol=1e-13), f"chunk {chunk} {dtype}"


# ---------------------------------------------------------------- cache operations
def pin_reshape_and_cache(L=None):
    """Token t's rows land at cache[slot // bs][h][slot % bs]; padding (slot < 0)
    and out-of-range slots write nothing; every other byte is untouched."""
    rng = np.random.default_rng(20)
    for dtype in DTYPES:
        NB, Hkv, bs, D, T = 10, 3, 4, 64, 14
        kc = H.poison((NB, Hkv, bs, D), dtype)
        vc = H.poison((NB, Hkv, bs, D), dtype)
        slots = rng.permutation(NB * bs)[:T].astype(np.int64)
        slots[3] = -1
        slots[7] = NB * bs + 5   # out of range
        k = _rand_store(rng, (T, Hkv, D), dtype)
        v = _rand_store(rng, (T, Hkv, D), dtype)
        bad = oracle.reshape_and_cache(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D,
                                       block_size=bs, dtype=dtype, L=L)
        assert bad == 1, "out-of-range slot count"
        written = 0
        for t in range(T):
            s = slots[t]
            if 0 <= s < NB * bs:
                assert np.array_equal(kc[s // bs, :, s % bs, :], k[t]), f"k row {t} {dtype}"
                assert np.array_equal(vc[s // bs, :, s % bs, :], v[t]), f"v row {t} {dtype}"
                written += 1
        untouched = NB * Hkv * bs * D - written * Hkv * D
        assert H.is_poison(kc).sum() == untouched and H.is_poison(vc).sum() == untouched, \
            f"bytes outside the slots changed {dtype}"


def pin_copy_blocks(L=None):
    """Block dst of both pools becomes a copy of block src; all else unchanged."""
    rng = np.random.default_rng(21)
    for dtype in DTYPES:
        NB, Hkv, bs, D = 12, 3, 8, 64
        kc = _rand_store(rng, (NB, Hkv, bs, D), dtype)
        vc = _rand_store(rng, (NB, Hkv, bs, D), dtype)
        k0, v0 = kc.copy(), vc.copy()
        pairs = np.array([[3, 7], [1, 2], [5, 0], [4, NB]], np.int64)
        bad = oracle.copy_blocks(kc, vc, pairs, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                 dtype=dtype, L=L)
        assert bad == 1, "bad pair count"
        ek, ev = k0.copy(), v0.copy()
        for s, d in pairs[:3]:
            ek[d], ev[d] = k0[s], v0[s]
        assert np.array_equal(kc, ek) and np.array_equal(vc, ev), f"copy_blocks {dtype}"


# ---------------------------------------------------------------- fp8 (E4M3) cache
def _torch_e4m3_values():
    """All 256 codes decoded by PyTorch's float8_e4m3fn (float64)."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e4m3_encode(x32: np.ndarray) -> np.ndarray:
    """binary32 values (|x| <= 448) -> codes by PyTorch's conversion."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


@np.errstate(invalid="ignore")
def pin_e4m3_codec(L=None):
    ref = _torch_e4m3_values()
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes, L)
    assert np.array_equal(got, ref, equal_nan=True), "e4m3 decode table"
    finite = ~np.isnan(ref)
    assert np.array_equal(oracle.encode_e4m3(ref[finite], L), codes[finite]), "e4m3 round trip"
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.05,
                        rng.uniform(-2.0 ** -6, 2.0 ** -6, 2000)]).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(x.astype(np.float64), L), _torch_e4m3_encode(x)), "e4m3 rounding"
    # exact midpoints between neighbouring positive codes go to the even code
    pos = [c for c in range(0x7e)]
    mids = np.array([(ref[c] + ref[c + 1]) / 2 for c in pos])
    want = np.array([c if c % 2 == 0 else c + 1 for c in pos], dtype=np.uint8)
    assert np.array_equal(oracle.encode_e4m3(mids, L), want), "e4m3 ties to even"
    assert np.array_equal(oracle.encode_e4m3(-mids, L), want | 0x80), "e4m3 negative ties"
    sat = oracle.encode_e4m3(np.array([449.0, 1e6, np.inf, -460.0, -np.inf]), L)
    assert np.array_equal(sat, np.array([0x7e, 0x7e, 0x7e, 0xfe, 0xfe], dtype=np.uint8)), "e4m3 saturation"


def pin_fp8_attention(L=None):
    """Power-of-two scales make scale * code exact in binary32, so attention
    over E4M3 pools must equal, bit for bit, the binary32 oracle over pools
    holding those values (and a binary32 copy of the binary16 queries)."""
    rng = np.random.default_rng(33)
    B, H_, Hkv, D, bs, NB = 3, 4, 2, 16, 4, 20
    lens = np.array([1, 7, 13], dtype=np.int32)
    _, kc16, vc16, bt, lens = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, "f16")
    finite = np.flatnonzero(~np.isnan(_torch_e4m3_values()))
    kc8 = rng.choice(finite, size=kc16.shape).astype(np.uint8)
    vc8 = rng.choice(finite, size=vc16.shape).astype(np.uint8)
    q = _rand_store(rng, (B, H_, D), "f16")
    vals = _torch_e4m3_values()
    for ks, vs in ((1.0, 1.0), (0.5, 2.0 ** -3)):
        kc32 = (vals[kc8] * ks).astype(np.float32)
        vc32 = (vals[vc8] * vs).astype(np.float32)
        q32 = q.view(np.float16).astype(np.float32)
        ref = oracle.paged_attention(q32, kc32, vc32, bt, lens, scale=0.3, num_heads=H_, num_kv_heads=Hkv,
                                     head_dim=D, block_size=bs, dtype="f32", L=L)
        got = oracle.paged_attention_fp8(q, kc8, vc8, bt, lens, scale=0.3, k_scale=ks, v_scale=vs, num_heads=H_,
                                         num_kv_heads=Hkv, head_dim=D, block_size=bs, q_dtype="f16", L=L)
        assert np.array_equal(got, ref), f"fp8 attention (scales {ks}, {vs})"


def pin_fp8_cache_write(L=None):
    """Each element lands at its slot as the E4M3 rounding of the binary32
    quotient x / scale (numpy's float32 division, PyTorch's rounding)."""
    rng = np.random.default_rng(35)
    T, Hkv, D, bs, NB = 9, 2, 16, 4, 8
    for dtype in ("f16", "bf16"):
        k = _rand_store(rng, (T, Hkv, D), dtype)
        v = _rand_store(rng, (T, Hkv, D), dtype)
        slots = rng.permutation(NB * bs)[:T].astype(np.int64)
        slots[2] = -1
        kc = rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8)
        vc = kc.copy()
        kc0, vc0 = kc.copy(), vc.copy()
        ks, vs = np.float32(0.037), np.float32(0.011)
        bad = oracle.reshape_and_cache_fp8(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                           src_dtype=dtype, k_scale=float(ks), v_scale=float(vs), L=L)
        assert bad == 0
        ek, ev = kc0.copy(), vc0.copy()
        for t in range(T):
            if slots[t] < 0:
                continue
            b, r = slots[t] // bs, slots[t] % bs
            ek[b, :, r, :] = _torch_e4m3_encode(_dec(k[t], dtype).astype(np.float32) / ks)
            ev[b, :, r, :] = _torch_e4m3_encode(_dec(v[t], dtype).astype(np.float32) / vs)
        assert np.array_equal(kc, ek) and np.array_equal(vc, ev), f"fp8 cache write ({dtype})"


# ---------------------------------------------------------------- 4-bit (q4_0) cache
def _f16_of_bits(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _q4_row_values(row: np.ndarray, D: int) -> np.ndarray:
    """Reference read-back of one q4_0 cache row with numpy, from the row
    layout: D/32 binary16 scales, then 16 code bytes per block whose byte j
    holds element j (low four bits) and element j + 16 (high four bits)."""
    nb = D // 32
    d = _f16_of_bits(row[:2 * nb].view(np.uint16))
    codes = row[2 * nb:].reshape(nb, 16)
    q = np.concatenate([codes & 0xF, codes >> 4], axis=1).astype(np.float64)  # [nb][32]
    return ((q - 8.0) * d[:, None]).reshape(-1)


@np.errstate(over="ignore")
def pin_f16_encoder(L=None):
    """The binary16 rounding of the scale against numpy's float32 -> float16
    conversion: nearest, ties to even, subnormals, overflow to infinity."""
    rng = np.random.default_rng(61)
    x = [rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000), rng.uniform(-2.0 ** -14, 2.0 ** -14, 1000),
         np.array([65504.0, 65519.0, 65520.0, 7e4, -1e6, 0.0, -0.0, 2.0 ** -25, 1.5 * 2.0 ** -24, 2.0 ** -26])]
    pos = np.arange(0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2  # exact in binary32 (12 significant bits)
    x += [mids[::7], -mids[::11]]
    x32 = np.concatenate(x).astype(np.float32)
    want = x32.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode_f16(x32.astype(np.float64), L), want), "binary16 rounding"


def pin_q4_0_exact_blocks(L=None):
    """Blocks x_j = d (k_j - 8) with integers k_j in [0, 15], k_0 = 0 and d a
    power of two: -8 d is the first element of largest magnitude, so the
    scale is d, every x_j / d + 8.5 = k_j + 0.5 is exact, the codes are the
    k_j themselves, and the block reads back exactly."""
    rng = np.random.default_rng(63)
    for e in (-12, -3, 0, 5, 11):
        for sgn in (1.0, -1.0):
            d = sgn * 2.0 ** e
            k = rng.integers(0, 16, 64)
            k[0] = k[32] = 0
            x = d * (k - 8.0)
            d_bits, qs = oracle.q4_0_quantize_block(x[:32].astype(np.float32), L)
            assert _f16_of_bits(d_bits) == d, f"q4_0 scale (d = {d})"
            want = (k[:16] | (k[16:32] << 4)).astype(np.uint8)
            assert np.array_equal(qs, want), f"q4_0 codes and nibble order (d = {d})"
            # the same values as a binary16 row of two blocks
            src = x.astype(np.float16).view(np.uint16)
            row = oracle.q4_0_quantize_row(src, "f16", L)
            assert row.shape == (36,) and np.array_equal(row[:4].view(np.uint16), np.array([d_bits, d_bits]))
            assert np.array_equal(_q4_row_values(row, 64), x), f"q4_0 exact read-back (d = {d})"
            assert np.array_equal(oracle.q4_0_values(row, 64, L), x), f"q4_0 oracle read-back (d = {d})"


def pin_q4_0_rules(L=None):
    """Hand-derived blocks for the rules of the format's reading.
    (a) Ties in magnitude go to the first element: x_0 = -1, x_5 = +1, the
        rest 0.25: m = -1, d = 0.125, x / d + 8.5 gives 0.5, 16.5 and 10.5,
        so codes 0, 15 (clamped) and 10; scale bits 0x3000.
    (b) Codes round half up: with d = 1 (x_0 = -8), 0.5 -> 9.0 -> code 9,
        -0.5 -> 8.0 -> 8, 1.5 -> 10.0 -> 10, -1.5 -> 7.0 -> 7.
    (c) A zero block: m = +0, d = -0 (scale bits 0x8000), every code 8."""
    x = np.full(32, 0.25, dtype=np.float32)
    x[0], x[5] = -1.0, 1.0
    d_bits, qs = oracle.q4_0_quantize_block(x, L)
    want = np.full(16, 0xAA, dtype=np.uint8)
    want[0], want[5] = 0xA0, 0xAF
    assert d_bits == 0x3000 and np.array_equal(qs, want), "q4_0 first maximum, clamp"
    x = np.zeros(32, dtype=np.float32)
    x[0], x[1], x[2], x[3], x[4] = -8.0, 0.5, -0.5, 1.5, -1.5
    d_bits, qs = oracle.q4_0_quantize_block(x, L)
    codes = np.concatenate([qs & 0xF, qs >> 4])
    assert d_bits == 0x3C00 and list(codes[:5]) == [0, 9, 8, 10, 7] and np.all(codes[5:] == 8), \
        "q4_0 rounding half up"
    d_bits, qs = oracle.q4_0_quantize_block(np.zeros(32, dtype=np.float32), L)
    assert d_bits == 0x8000 and np.all(qs == 0x88), "q4_0 zero block"


def pin_q4_0_error_bound(L=None):
    """Random rows (normal, heavy-tailed, tiny, bfloat16): every value reads
    back within |d| (1 + 2^-7) of itself (half a step, or one step where the
    code saturates at 15, plus the binary16 rounding of d), and the element of
    largest magnitude of each block within |m| 2^-11 (its code is 0)."""
    rng = np.random.default_rng(65)
    for dtype, scale in (("f16", 1.0), ("f16", 3e-4), ("bf16", 50.0)):
        for _ in range(40):
            D = 128
            raw = rng.standard_normal(D) * scale
            raw[rng.integers(0, D, 3)] *= 30.0
            src = H.round_to_storage(raw, dtype)
            x = _dec(src, dtype)
            row = oracle.q4_0_quantize_row(src, dtype, L)
            got = _q4_row_values(row, D)
            d = np.abs(_f16_of_bits(row[:8].view(np.uint16)))
            for b in range(4):
                xb, gb = x[32 * b:32 * b + 32], got[32 * b:32 * b + 32]
                assert np.all(np.abs(xb - gb) <= d[b] * (1 + 2.0 ** -7)), "q4_0 error bound"
                j = int(np.argmax(np.abs(xb)))
                assert abs(gb[j] - xb[j]) <= abs(xb[j]) * 2.0 ** -11, "q4_0 largest element"


def pin_q4_0_cache_write(L=None):
    """Each (token, kv head) row lands at its slot as that row's q4_0 bytes;
    a negative slot is skipped, an out-of-range one counted; every other
    byte of the pools is untouched."""
    rng = np.random.default_rng(67)
    T, Hkv, D, bs, NB = 9, 2, 64, 4, 8
    rb = oracle.q4_0_row_bytes(D)
    for dtype in ("f16", "bf16"):
        k = _rand_store(rng, (T, Hkv, D), dtype)
        v = _rand_store(rng, (T, Hkv, D), dtype, scale=0.1)
        slots = rng.permutation(NB * bs)[:T].astype(np.int64)
        slots[2], slots[4] = -1, NB * bs + 3
        kc = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
        vc = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
        ek, ev = kc.copy(), vc.copy()
        bad = oracle.reshape_and_cache_q4_0(k, v, kc, vc, slots, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                            src_dtype=dtype, L=L)
        assert bad == 1, "q4_0 out-of-range slot count"
        for t in range(T):
            if slots[t] < 0 or slots[t] >= NB * bs:
                continue
            b, r = slots[t] // bs, slots[t] % bs
            for h in range(Hkv):
                ek[b, h, r] = oracle.q4_0_quantize_row(np.ascontiguousarray(k[t, h]), dtype, L)
                ev[b, h, r] = oracle.q4_0_quantize_row(np.ascontiguousarray(v[t, h]), dtype, L)
        assert np.array_equal(kc, ek) and np.array_equal(vc, ev), f"q4_0 cache write ({dtype})"


def pin_q4_0_attention(L=None):
    """Every q4_0 value d (q - 8) is exact in binary32, so attention over q4_0
    pools must equal, bit for bit, the binary32 oracle over pools holding the
    values numpy reads back from the rows."""
    rng = np.random.default_rng(69)
    B, H_, Hkv, D, bs, NB = 3, 4, 2, 64, 4, 20
    lens = np.array([1, 7, 13], dtype=np.int32)
    _, kc16, _, bt, lens = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, "f16")
    rb = oracle.q4_0_row_bytes(D)

    def pool(sc):
        p = rng.integers(0, 256, (NB, Hkv, bs, rb), dtype=np.uint8)
        sbits = (rng.standard_normal((NB, Hkv, bs, D // 32)) * sc).astype(np.float16).view(np.uint16)
        p[..., :D // 16] = sbits.view(np.uint8).reshape(NB, Hkv, bs, D // 16)
        vals = np.stack([_q4_row_values(r, D) for r in p.reshape(-1, rb)]).reshape(NB, Hkv, bs, D)
        return p, vals.astype(np.float32)

    kq, k32 = pool(0.05)
    vq, v32 = pool(0.3)
    q = _rand_store(rng, (B, H_, D), "f16")
    q32 = q.view(np.float16).astype(np.float32)
    ref = oracle.paged_attention(q32, k32, v32, bt, lens, scale=0.3, num_heads=H_, num_kv_heads=Hkv, head_dim=D,
                                 block_size=bs, dtype="f32", L=L)
    got = oracle.paged_attention_q4_0(q, kq, vq, bt, lens, scale=0.3, num_heads=H_, num_kv_heads=Hkv, head_dim=D,
                                      block_size=bs, q_dtype="f16", L=L)
    assert np.array_equal(got, ref), "q4_0 attention"


# ---------------------------------------------------------------- paged prefill
def _prefill_case(rng, dtype="f16"):
    B, H_, Hkv, D, bs, NB = 3, 4, 2, 16, 4, 40
    lens = np.array([1, 9, 22], dtype=np.int32)
    q_unused, kc, vc, bt, lens = _random_paged(rng, B, H_, Hkv, D, bs, NB, lens, dtype)
    return B, H_, Hkv, D, bs, kc, vc, bt, lens


def pin_prefill_single_query_is_decode(L=None):
    rng = np.random.default_rng(51)
    B, H_, Hkv, D, bs, kc, vc, bt, lens = _prefill_case(rng)
    q = _rand_store(rng, (B, H_, D), "f16")
    qs = np.arange(B + 1, dtype=np.int32)
    got = oracle.paged_prefill(q, kc, vc, bt, lens, qs, scale=0.4, num_heads=H_, num_kv_heads=Hkv, head_dim=D,
                               block_size=bs, dtype="f16", L=L)
    ref = _attn(L, q, kc, vc, bt, lens, H_, Hkv, D, bs, "f16", 0.4)
    assert np.array_equal(got, ref), "one-query prefill == decode"


def pin_prefill_prefix_dense(L=None):
    """Query i of sequence s (context L_s, n_s queries) sits at position
    L_s - n_s + i and must equal dense attention over exactly the tokens
    0 .. that position, gathered with numpy from the block table."""
    rng = np.random.default_rng(53)
    B, H_, Hkv, D, bs, kc, vc, bt, lens = _prefill_case(rng)
    n = np.array([1, 4, 22], dtype=np.int32)  # the last sequence is a full prompt
    qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = _rand_store(rng, (int(qs[-1]), H_, D), "f16")
    got = oracle.paged_prefill(q, kc, vc, bt, lens, qs, scale=0.4, num_heads=H_, num_kv_heads=Hkv, head_dim=D,
                               block_size=bs, dtype="f16", L=L)
    ks, vs, starts = [], [], [0]
    for s in range(B):
        for i in range(int(n[s])):
            pos = int(lens[s]) - int(n[s]) + i
            t = np.arange(pos + 1)
            ks.append(kc[bt[s, t // bs], :, t % bs, :])
            vs.append(vc[bt[s, t // bs], :, t % bs, :])
            starts.append(starts[-1] + pos + 1)
    ref = oracle.dense_attention(q, np.ascontiguousarray(np.concatenate(ks)), np.ascontiguousarray(np.concatenate(vs)),
                                 np.array(starts, dtype=np.int64), scale=0.4, num_heads=H_, num_kv_heads=Hkv,
                                 head_dim=D, dtype="f16", L=L)
    assert np.array_equal(got, ref), "prefill query == dense attention over its prefix"


ALL_PINS = [pin_decoders, pin_context_one, pin_uniform_weights, pin_dominant_logit,
            pin_two_tokens, pin_gqa_mapping, pin_brute_force, pin_dense_equivalence,
            pin_placement_invariance, pin_copy_on_write, pin_split_merge,
            pin_reshape_and_cache, pin_copy_blocks, pin_e4m3_codec, pin_fp8_attention,
            pin_fp8_cache_write, pin_prefill_single_query_is_decode, pin_prefill_prefix_dense,
            pin_f16_encoder, pin_q4_0_exact_blocks, pin_q4_0_rules, pin_q4_0_error_bound, pin_q4_0_cache_write,
            pin_q4_0_attention]
